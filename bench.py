"""Benchmark of the KVarN 2-bit KV-cache hot path on GB300.

One step = one decode step of the Qwen3-4B-shaped full cache: for each of the
36 layers, the append of every sequence's new token (which completes the
open 64-token block and quantises it into the paged pool) followed by decode
attention over the 2-bit cache (8192 tokens x 64 sequences x 8 kv heads,
physical blocks randomly permuted per layer). The per-step cache (16.3 GB)
is far larger than L2, so no flush is needed between steps.

Prints one JSON line (see the keys below). --impl reference times the fp64
CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "2-bit KV decode-attn GB/s (% of HBM peak) + quantize-append tokens/s"
CPU_SAMPLE_SEQS = 16
FALLBACK_HBM_GBS = 6800.0
D = 128


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    p.add_argument("--layers", type=int, default=None, help="(testing only) fewer layers")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-bf16", action="store_true")
    p.add_argument("--ablation", action="store_true",
                   help="instead of the step: error of each ablation (Hadamard only, VarN only, one VarN "
                        "axis) against the bf16 cache on the Llama-3.1-8B layer, one JSON line per variant")
    p.add_argument("--prefill", action="store_true",
                   help="instead of the step: chunked prefill attention over the Llama-3.1-8B layer "
                        "(batch 16 x 4096 cached tokens) for several chunk lengths, one JSON line each")
    p.add_argument("--llama-layer", action="store_true",
                   help="instead of the step: the Llama-3.1-8B layer (batch 16 x 4096, block 32): one append "
                        "that completes every open block, then decode attention; each rep after an "
                        "L2-flushing write, median; one JSON line")
    p.add_argument("--long", action="store_true",
                   help="instead of the step: the Phi-4-14B long-horizon workload (40 layers, batch 8, "
                        "prefill 1024-2048 then 16384 x (append + attention) per layer): us per step over "
                        "the horizon and the 2-bit vs bf16-cache output error at steps 1 .. 16384")
    p.add_argument("--long-steps", type=int, default=16384, help="appends per layer in --long")
    p.add_argument("--long-eager", action="store_true",
                   help="with --long: every step as eager calls (no CUDA graph after the first window)")
    p.add_argument("--sweep", action="store_true",
                   help="instead of the step: the Llama-3.1-8B layer grid (batch x context, ragged "
                        "lengths), 2-, 3- and 4-bit vs bf16-cache decode attention, one JSON line per point")
    p.add_argument("--point", type=int, nargs=2, metavar=("BATCH", "CTX"),
                   help="with --sweep: only this grid point")
    return p.parse_args()


# ---------------------------------------------------------------------------- ranks

def barrier():
    """torch.distributed barrier when a process group is up (N > 1), else nothing."""
    import torch.distributed as tdist
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        tdist.barrier()


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest of every rank's x (the slowest rank's time); x itself at N = 1.
    `device` is where the one-element tensor lives: the GPU under NCCL, the
    host under gloo."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    barrier()
    return float(t.item())


def whole_job_gbs(bytes_per_rank: float, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank moves bytes_per_rank per step; the job's step
    time is the slowest rank's."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def workload():
    import synth
    return synth.QWEN3_4B_CACHE


def algorithmic_bytes(w, layers):
    """Bytes the step must move at minimum: the algorithmic bytes of the roofline."""
    B, n_kv, n_q, batch, L = w.block, w.n_kv, w.n_q, w.batch, w.ctx
    per_token_head = 2 * (32 + 16 + 2) + 2 * 256 / B          # K+V: codes, s/z, R + C share
    attn_cache = batch * L * n_kv * per_token_head
    attn_other = batch * n_q * (D * 2 + D * 4) + batch * (L // B) * 4   # q bf16, out fp32, table
    attn = attn_cache + attn_other
    # append: new rows in (bf16), the open block's staged rows read, packed block written
    hb = 50 * B + 256
    app = batch * n_kv * 2 * (D * 2 + (B - 1) * D * 2 + hb)
    return attn * layers, app * layers, attn, app


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def attention_source_hash():
    """SHA-256 of the attention kernel's sources with comments and blank lines
    removed (a comment edit does not change the kernel the counters describe)."""
    import re
    h = hashlib.sha256()
    for f in ("attention.cu", "attn_common.cuh", "split.cuh", "common.cuh"):
        text = open(os.path.join(ROOT, "bit_kv_cache_08_gb300", "csrc", f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()


def _attention_record():
    """profiles/attention_traffic.json (ncu counters of one attention launch on
    the Qwen3-4B layer) if it was captured from the current kernel source."""
    path = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    return rec if rec.get("source_sha256") == attention_source_hash() else None


def traffic_record():
    """ncu DRAM bytes per attention launch, valid only for the kernel source it
    was captured from."""
    rec = _attention_record()
    return rec.get("bytes_per_launch") if rec else None


def issue_context(attn_launch_ms, sm_mhz, sms):
    """The attention kernel against the instruction-issue ceiling: warp
    instructions of one split-K launch (ncu, current source only) over the
    live split + merge time, against 4 issues per SM and cycle at the sampled
    SM clock."""
    rec = _attention_record()
    n = rec.get("split_kernel", {}).get("warp_instr") if rec else None
    if not n or not sm_mhz or not sms:
        return None
    achieved = n / (attn_launch_ms * 1e-3)
    peak = sms * 4 * sm_mhz * 1e6
    return {"warp_instr_per_launch": int(n), "achieved_warp_instr_per_s": round(achieved / 1e12, 4),
            "peak_warp_instr_per_s": round(peak / 1e12, 4), "unit": "T warp-instr/s",
            "frac": round(achieved / peak, 4),
            "note": "context for the HBM roofline: the kernel is bound by instruction issue"}


class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.idx = device_index
        # the raw samples go to $KVARN_CLOCKS_DIR (kept for inspection) or the temp directory
        d = os.environ.get("KVARN_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            # wait (outside the timed region) until the sampler is live
            t_end = time.time() + 3.0
            while time.time() < t_end and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- GPU arm

def build_layers(kv, w, layers, device):
    """Prefill every layer's 2-bit cache to ctx-1 tokens (ctx-1 = 8191: 127
    full blocks in the pool, 63 rows in staging); per-layer permuted tables."""
    import numpy as np
    import torch
    import synth
    B, n_kv, batch, L = w.block, w.n_kv, w.batch, w.ctx
    nb = L // B
    state = []
    for layer in range(layers):
        sb = synth.sign_bits(1000 + layer)
        cfg = kv.make_config(w.n_q, n_kv, B, w.iters, sb)
        g = synth.make_gen(w.seed * 1000 + layer, device)
        pool = kv.alloc_pool(cfg, batch * nb, device)
        staging = kv.alloc_staging(cfg, batch, device)
        ws0 = kv.alloc_workspace(cfg, 0, 0, device)
        perm = np.random.default_rng([w.seed, layer]).permutation(batch * nb).astype(np.int32)
        bt = torch.from_numpy(perm.reshape(batch, nb)).to(device)
        hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
        jj = torch.arange(nb - 1, device=device)
        for kind in (0, 1):
            T = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, device).to(torch.bfloat16)
            # every full block of every (sequence, head) in one call: offsets from the table
            src = T[:, :, :(nb - 1) * B].contiguous()                   # [batch][n_kv][(nb-1)B][128]
            offs = (bt[:, None, :nb - 1].long() * bb + (2 * torch.arange(n_kv, device=device)[None, :, None] + kind)
                    * hb).reshape(-1).contiguous()
            kv.quantize_block(cfg, kind, src, pool, ws0, dst_offsets=offs, n_head_blocks=offs.numel())
            staging[:, :, kind, :B - 1] = T[:, :, (nb - 1) * B:L - 1]
            if kind == 0:
                k_last = T[:, :, L - 1].contiguous()
            else:
                v_last = T[:, :, L - 1].contiguous()
            del T, src
        torch.cuda.synchronize()
        assert kv.read_error(ws0) == 0
        q = synth.queries(g, batch, w.n_q, device).to(torch.bfloat16)
        state.append(dict(cfg=cfg, pool=pool, staging=staging, bt=bt, q=q, k_new=k_last, v_new=v_last))
        del jj
    return state


def run_gpu(args, rank, world):
    import torch
    import bit_kv_cache_08_gb300 as kv
    kv.build()
    local = int(os.environ.get("LOCAL_RANK", rank))
    device = f"cuda:{local % max(1, torch.cuda.device_count())}"
    torch.cuda.set_device(device)
    w = workload()
    layers = args.layers or w.layers
    state = build_layers(kv, w, layers, device)
    B, batch = w.block, w.batch
    nb = w.ctx // B
    cfg0 = state[0]["cfg"]
    ws = kv.alloc_workspace(cfg0, batch, nb, device)
    pos = torch.full((batch,), w.ctx - 1, dtype=torch.int32, device=device)
    lens = torch.full((batch,), w.ctx, dtype=torch.int32, device=device)
    out = torch.empty(layers, batch, w.n_q, D, device=device)

    def step(events=None):
        for l, st in enumerate(state):
            if events is not None:
                events[l][0].record()
            kv.append(st["cfg"], st["pool"], st["staging"], st["bt"], pos, st["k_new"], st["v_new"], ws)
            if events is not None:
                events[l][1].record()
            kv.decode_attn(st["cfg"], st["q"], st["pool"], st["staging"], st["bt"], lens, out[l], ws)
            if events is not None:
                events[l][2].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0, "device error during warm-up"

    # per-kernel breakdown: the eager loop with CUDA events around every launch
    attn_ms, app_ms = [], []
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(layers)]
           for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(args.steps):
        step(evs[s])
    e1.record()
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, device)
    for s in range(args.steps):
        for l in range(layers):
            e = evs[s][l]
            app_ms.append(e[0].elapsed_time(e[1]))
            attn_ms.append(e[1].elapsed_time(e[2]))
    assert kv.read_error(ws) == 0, "device error during the eager steps"

    # the timed steps: the whole step (every layer's append + attention) captured
    # once as a CUDA graph and replayed K times (the same launches, no per-launch
    # host work); the eager loop stands in only if capture is refused here
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
        timing = "CUDA graph of the whole step replayed per step"
    except RuntimeError as e:
        graph = None
        timing = f"eager launches (graph capture failed: {e})"
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step()
        t1.record()
        torch.cuda.synchronize()
    barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), device)
    assert kv.read_error(ws) == 0, "device error during the timed steps"
    clocks = clk.summary()
    del graph
    attn_bytes, app_bytes, attn_launch_bytes, app_launch_bytes = algorithmic_bytes(w, layers)
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(attn_bytes + app_bytes, world, ms_per_step)
    attn_launch_ms = sum(attn_ms) / len(attn_ms)
    achieved = attn_launch_bytes / (attn_launch_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    app_launch_ms = sum(app_ms) / len(app_ms)
    appended_tokens = batch * layers            # per step: one token per sequence per layer
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded lognormal token scales, outlier channels; no weights or datasets)",
        "config": {"workload": w.name, "layers": layers, "batch": batch, "seq_len": w.ctx,
                   "n_q_heads": w.n_q, "n_kv_heads": w.n_kv, "head_dim": D, "block": B, "varn_iters": w.iters,
                   "step": "per layer: kvarn_append (completes every open block) + kvarn_decode_attn",
                   "l2": "no flush: per-step cache 16.3 GB >> 129 MB L2",
                   "parallelism": f"replicas x{world} (each rank its own {batch} sequences; no collective "
                                  "on the data path)"},
        "timing": timing,
        "decode_step_tokens_per_s": round(world * batch / (ms_per_step * 1e-3), 1),
        "eager_step": {"ms_per_step": round(eager_ms, 4),
                       "GB_per_s": round(whole_job_gbs(attn_bytes + app_bytes, world, eager_ms), 2),
                       "note": "the same step launched eagerly, CUDA events around every launch "
                               "(the per-kernel figures below)"},
        "decode_attn": {"GB_per_s": round(achieved, 1), "us_per_layer": round(attn_launch_ms * 1e3, 2),
                        "algorithmic_bytes_per_layer": int(attn_launch_bytes),
                        "frac_of_hbm_peak": round(achieved / peak, 4),
                        "tokens_per_s": round(world * batch * layers / (ms_per_step * 1e-3), 1)},
        "append": {"tokens_per_s": round(world * appended_tokens * w.n_kv * 2 / (sum(app_ms) * 1e-3 / args.steps), 1),
                   "seq_tokens_per_s": round(world * appended_tokens / (sum(app_ms) * 1e-3 / args.steps), 1),
                   "us_per_layer": round(app_launch_ms * 1e3, 2),
                   "algorithmic_bytes_per_layer": int(app_launch_bytes),
                   "GB_per_s": round(app_launch_bytes / (app_launch_ms * 1e-3) / 1e9, 1),
                   "frac_of_hbm_peak": round(app_launch_bytes / (app_launch_ms * 1e-3) / 1e9 / peak, 4),
                   "note": "tokens_per_s counts (sequence, layer, kv head, K|V) rows quantised"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic_record(),
                     "kernel": "kvarn_decode_attn (split-K kernel + merge), one layer",
                     "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "gpu_launches": args.steps * layers * 3,
        "clocks": clocks,
    }
    res["issue"] = issue_context(attn_launch_ms, clocks.get("sm_mhz") if isinstance(clocks, dict) else None,
                                 torch.cuda.get_device_properties(device).multi_processor_count)
    return res, state, (kv, ws, pos, lens, out)


def e2e_gpu(args, ctx_objs, state, w, world):
    """The same step through the C ABI with host buffers: every step copies the
    step's queries and new K/V rows from pinned host memory and reads the
    outputs back, each layer's copies overlapped with the other layers'
    kernels."""
    import torch
    kv, ws, pos, lens, out = ctx_objs
    layers = len(state)
    # one pinned row per layer holding its q, new K and new V back to back (one
    # copy per layer); the device tensors the API gets are views of its copy
    sq, sk = state[0]["q"].shape, state[0]["k_new"].shape
    nq, nk = state[0]["q"].numel(), state[0]["k_new"].numel()
    hbuf = torch.empty(layers, nq + 2 * nk, dtype=state[0]["q"].dtype).pin_memory()
    for l, st in enumerate(state):
        hbuf[l, :nq] = st["q"].reshape(-1).cpu()
        hbuf[l, nq:nq + nk] = st["k_new"].reshape(-1).cpu()
        hbuf[l, nq + nk:] = st["v_new"].reshape(-1).cpu()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dbuf = hbuf.to(out.device)
    dq = [dbuf[l, :nq].view(sq) for l in range(layers)]
    dk = [dbuf[l, nq:nq + nk].view(sk) for l in range(layers)]
    dv = [dbuf[l, nq + nk:].view(sk) for l in range(layers)]

    # copies on their own streams, overlapped with the layers' kernels: layer l
    # waits for its inputs only, and its output goes back while the next layers run
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(layers)]
    ev_out = [torch.cuda.Event() for _ in range(layers)]

    def step():
        main = torch.cuda.current_stream()
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        with torch.cuda.stream(s_in):
            for l in range(layers):
                dbuf[l].copy_(hbuf[l], non_blocking=True)
                ev_in[l].record(s_in)
        # copies on one stream finish in order: layer 0 waits for the first three
        # layers' inputs and layer 3 for all of them, long copied by then (fewer
        # cross-stream waits between the layers' kernels)
        waits = {0: ev_in[min(2, layers - 1)]}
        if layers > 3:
            waits[3] = ev_in[layers - 1]
        for l, st in enumerate(state):
            if l in waits:
                main.wait_event(waits[l])
            kv.append(st["cfg"], st["pool"], st["staging"], st["bt"], pos, dk[l], dv[l], ws)
            kv.decode_attn(st["cfg"], dq[l], st["pool"], st["staging"], st["bt"], lens, out[l], ws)
            ev_out[l].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_out[l])
                hout[l].copy_(out[l], non_blocking=True)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    # the whole step (copies in, the API calls of every layer, copy out) captured
    # once as a CUDA graph and replayed, as a serving loop runs its decode step;
    # eager calls if capture fails
    graph, timing = None, "eager API calls"
    try:
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            step()
        torch.cuda.current_stream().wait_stream(cs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(max(1, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        timing = ("CUDA graph of the step (every layer's inputs copied in and its output copied out on "
                  "side streams, overlapped with the layers' API calls) replayed")
    except RuntimeError:
        graph = None
    run = graph.replay if graph is not None else step
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    ms = max_over_ranks(ms, out.device)
    attn_bytes, app_bytes, _, _ = algorithmic_bytes(w, layers)
    h2d = hbuf.numel() * hbuf.element_size()
    d2h = hout.numel() * 4
    return {"value": round(whole_job_gbs(attn_bytes + app_bytes, world, ms), 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "timing": timing + "; host clock around the K steps"}


def bf16_comparison(kv, w, device):
    """The repo's bf16-cache decode attention on one layer of the same shape."""
    import numpy as np
    import torch
    import synth
    B, n_kv, batch, L = w.block, w.n_kv, w.batch, w.ctx
    nb = L // B
    cfg = kv.make_config(w.n_q, n_kv, B, w.iters, synth.sign_bits(0))
    g = synth.make_gen(7, device)
    pool = torch.empty(batch * nb, n_kv, 2, B, D, dtype=torch.bfloat16, device=device)
    pool.normal_(generator=g)
    perm = np.random.default_rng(7).permutation(batch * nb).astype(np.int32)
    bt = torch.from_numpy(perm.reshape(batch, nb)).to(device)
    q = synth.queries(g, batch, w.n_q, device).to(torch.bfloat16)
    lens = torch.full((batch,), L, dtype=torch.int32, device=device)
    out = torch.empty(batch, w.n_q, D, device=device)
    ws = kv.alloc_workspace(cfg, batch, nb, device)
    for _ in range(3):
        kv.decode_attn_bf16(cfg, q, pool, bt, lens, out, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record()
    for _ in range(reps):
        kv.decode_attn_bf16(cfg, q, pool, bt, lens, out, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nbytes = batch * L * n_kv * 2 * D * 2 + batch * w.n_q * D * 6
    del pool
    return {"GB_per_s": round(nbytes / (ms * 1e-3) / 1e9, 1), "us_per_layer": round(ms * 1e3, 2),
            "tokens_per_s_per_layer": round(batch / (ms * 1e-3), 1),
            "bytes_per_layer": int(nbytes), "note": "same shape, bf16 pages, fp32 arithmetic"}


def bulk_quantize(kv, w, device, peak):
    """kvarn_quantize_block in prefill mode: every 64-token block of one
    layer's K (64 sequences x 8 kv heads x 8192 tokens, bf16, 1.07 GB in)
    quantised in one call into a contiguous scratch pool."""
    import torch
    import synth
    B, n_kv, batch, L = w.block, w.n_kv, w.batch, w.ctx
    cfg = kv.make_config(w.n_q, n_kv, B, w.iters, synth.sign_bits(3))
    g = synth.make_gen(11, device)
    src = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, device).to(torch.bfloat16)
    n = batch * n_kv * (L // B)
    hb = kv.head_block_bytes(cfg)
    dst = torch.empty(n * hb, dtype=torch.uint8, device=device)
    ws = kv.alloc_workspace(cfg, 0, 0, device)
    for _ in range(3):
        kv.quantize_block(cfg, 0, src, dst, ws, n_head_blocks=n)
    torch.cuda.synchronize()
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        kv.quantize_block(cfg, 0, src, dst, ws, n_head_blocks=n)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    assert kv.read_error(ws) == 0
    ms = statistics.median(ts)
    rows = n * B
    nbytes = rows * D * 2 + n * hb
    del src, dst
    return {"head_rows_per_s": round(rows / (ms * 1e-3), 1), "GB_per_s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "us_per_call": round(ms * 1e3, 1),
            "head_blocks": n, "bytes": int(nbytes),
            "note": "one call over a layer's K: 256 B in + 54 B out per (token, kv head) row; "
                    "bound by instruction issue, not HBM"}


# ---------------------------------------------------------------------------- oracle (CPU)

def cpu_sample_setup(w, seqs, seed=0):
    """A bounded sample of the workload for the fp64 oracle: `seqs` sequences
    of one layer (all kv heads), with the cache as prefill left it (not
    timed). The timed step (cpu_sample_step) quantises the completed block of
    every (sequence, head, K|V), then runs decode attention over all tokens."""
    import numpy as np
    import torch
    import oracle
    import synth
    B, n_kv, L = w.block, w.n_kv, w.ctx
    nb = L // B
    sb = synth.sign_bits(1000)
    g = synth.make_gen(seed)
    K = synth.kv_values(g, seqs, n_kv, L, w.sigma_m, w.n_out, w.out_factor).to(torch.bfloat16)
    V = synth.kv_values(g, seqs, n_kv, L, w.sigma_m, w.n_out, w.out_factor).to(torch.bfloat16)
    q = synth.queries(g, seqs, w.n_q).to(torch.bfloat16).double().numpy()
    hb = oracle.head_block_bytes(B)
    pool = np.zeros((seqs * nb, n_kv, 2, hb), dtype=np.uint8)
    last = []
    for kind, T in ((0, K), (1, V)):
        X = T[:, :, :(nb - 1) * B].double().numpy().reshape(seqs, n_kv, nb - 1, B, D)
        qb = oracle.quantize_blocks(X.transpose(0, 2, 1, 3, 4).reshape(-1, B, D), w.iters, kind, sb)
        pool[np.arange(seqs)[:, None] * nb + np.arange(nb - 1)[None, :], :, kind] = \
            qb.reshape(seqs, nb - 1, n_kv, hb)
        last.append(np.ascontiguousarray(T[:, :, (nb - 1) * B:].double().numpy().reshape(seqs * n_kv, B, D)))
    bt = (np.arange(seqs)[:, None] * nb + np.arange(nb)[None, :]).astype(np.int32)
    return dict(w=w, seqs=seqs, sb=sb, q=q, pool=pool, last=last, bt=bt, hb=hb,
                staging=np.zeros((seqs, n_kv, 2, B, D), dtype=np.uint16),
                lens=np.full(seqs, L, dtype=np.int32))


def cpu_sample_step(st):
    """Returns (seconds, algorithmic bytes, threads) of one timed oracle step."""
    import numpy as np
    import oracle
    w, seqs, B, n_kv, L = st["w"], st["seqs"], st["w"].block, st["w"].n_kv, st["w"].ctx
    nb = L // B
    t0 = time.perf_counter()
    for kind in (0, 1):
        qb = oracle.quantize_blocks(st["last"][kind], w.iters, kind, st["sb"])
        st["pool"][np.arange(seqs) * nb + nb - 1, :, kind] = qb.reshape(seqs, n_kv, st["hb"])
    oracle.decode_attention(B, w.n_q, n_kv, st["sb"], 1 / math.sqrt(D), st["q"], st["pool"], st["staging"],
                            st["bt"], st["lens"])
    secs = time.perf_counter() - t0
    attn_bytes = seqs * L * n_kv * (2 * (32 + 16 + 2) + 2 * 256 / B) + seqs * w.n_q * D * 6
    app_bytes = seqs * n_kv * 2 * (D * 2 + (B - 1) * D * 2 + st["hb"])
    return secs, attn_bytes + app_bytes, oracle.max_threads()


def cpu_baseline(w):
    """The oracle timed on the host cores twice: with its OpenMP loops on all
    threads (16 sequences of one layer) and single-threaded (4 sequences)."""
    import oracle
    out = {}
    nthreads = oracle.max_threads()
    for key, threads, seqs in (("all", nthreads, CPU_SAMPLE_SEQS), ("single", 1, CPU_SAMPLE_SEQS // 4)):
        oracle.set_threads(threads)
        secs, nbytes, used = cpu_sample_step(cpu_sample_setup(w, seqs))
        out[key] = {"value": round(nbytes / secs / 1e9, 4), "cores": used, "seconds": round(secs, 2),
                    "sample": f"{seqs} of {w.batch} sequences x 1 of {w.layers} layers, all kv heads: "
                              f"block quantise + attention"}
    oracle.set_threads(nthreads)
    a = out["all"]
    return {"value": a["value"], "unit": "GB/s", "cores": a["cores"], "kind": "oracle",
            "sample": f"{a['sample']} ({a['seconds']} s)",
            "single_thread": {"value": out["single"]["value"], "unit": "GB/s", "cores": 1,
                              "sample": f"{out['single']['sample']} ({out['single']['seconds']} s)"},
            "nproc": os.cpu_count(), "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


def run_reference(args):
    w = workload()
    seqs = CPU_SAMPLE_SEQS
    st = cpu_sample_setup(w, seqs)
    secs_list = []
    nbytes = 0
    threads = 1
    for _ in range(args.warmup):
        cpu_sample_step(st)
    for _ in range(args.steps):
        s, nbytes, threads = cpu_sample_step(st)
        secs_list.append(s)
    secs = sum(secs_list) / len(secs_list)
    value = nbytes / secs / 1e9
    sample = (f"{seqs} of {w.batch} sequences x 1 of {w.layers} layers (all {w.n_kv} kv heads): "
              f"block quantise + attention")
    return {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "device": "host cores (the oracle runs on no GPU)", "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------- sweep

SWEEP_BATCH = (1, 8, 32, 128, 256)
SWEEP_CTX = (1024, 8192, 32768, 131072)


def _time_events(fn, reps, flush):
    """Median of `reps` launches of fn, each timed alone with CUDA events on the
    current stream. Before every launch a 1 GiB write flushes L2; it also keeps
    the GPU busy while the host queues the start event and the launch, so the
    events bracket device time only (not the host's launch latency)."""
    import torch
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def run_sweep(args):
    import numpy as np
    import torch
    import bit_kv_cache_08_gb300 as kv
    import synth
    kv.build()
    dev = "cuda"
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    for batch in ((args.point[0],) if args.point else SWEEP_BATCH):
        for ctx in ((args.point[1],) if args.point else SWEEP_CTX):
            w = synth.sweep_point(batch, ctx)
            B, n_kv, n_q = w.block, w.n_kv, w.n_q
            lens = np.array(w.seq_lens, dtype=np.int64)
            nbs = (lens + B - 1) // B
            max_blocks = int(nbs.max())
            g = synth.make_gen(w.seed + batch + ctx, dev)
            n_phys = int(nbs.sum())
            perm = np.random.default_rng([batch, ctx]).permutation(n_phys).astype(np.int32)
            bt_np = np.full((batch, max_blocks), -1, dtype=np.int32)
            o = 0
            for b in range(batch):
                bt_np[b, :nbs[b]] = perm[o:o + nbs[b]]
                o += nbs[b]
            bt = torch.from_numpy(bt_np).to(dev)
            sl = torch.from_numpy(lens.astype(np.int32)).to(dev)
            q = synth.queries(g, batch, n_q, dev).to(torch.bfloat16)
            out = torch.empty(batch, n_q, D, device=dev)
            big = ctx * batch >= 1 << 22
            reps = 5 if big else 30
            full = (lens // B) * B
            packed = {}
            for bits in (2, 3, 4):
                cfg = kv.make_config(n_q, n_kv, B, w.iters, synth.sign_bits(w.seed), bits=bits)
                ws = kv.alloc_workspace(cfg, batch, max_blocks, dev)
                # packed cache: valid head-blocks (512 quantised K and V tiles repeated)
                hb = kv.head_block_bytes(cfg)
                tile = torch.empty(2, 256, hb, dtype=torch.uint8, device=dev)
                for kind in (0, 1):
                    x = synth.kv_values(g, 1, 256, B, w.sigma_m, w.n_out, w.out_factor, dev)[0].to(torch.bfloat16)
                    kv.quantize_block(cfg, kind, x.contiguous(), tile[kind], kv.alloc_workspace(cfg, 0, 0, dev))
                pool = kv.alloc_pool(cfg, n_phys, dev).view(n_phys, n_kv, 2, hb)
                for c0 in range(0, n_phys, 1 << 15):
                    c1 = min(n_phys, c0 + (1 << 15))
                    idx = (torch.arange(c0 * n_kv, c1 * n_kv, device=dev) % 256).view(c1 - c0, n_kv)
                    pool[c0:c1, :, 0] = tile[0][idx]
                    pool[c0:c1, :, 1] = tile[1][idx]
                pool = pool.view(n_phys, -1)
                staging = kv.alloc_staging(cfg, batch, dev)
                staging.normal_(generator=g)
                nbytes = float((full * n_kv * (2 * (16 * bits + 16 + 2) + 2 * 256 / B)).sum()
                               + ((lens - full) * n_kv * 512).sum() + batch * n_q * 768 + nbs.sum() * 4)
                ms = _time_events(lambda: kv.decode_attn(cfg, q, pool, staging, bt, sl, out, ws), reps, flush)
                assert kv.read_error(ws) == 0
                packed[bits] = (ms, nbytes)
                del pool, staging
                torch.cuda.empty_cache()
            ms2, b2 = packed[2]
            ms3, b3 = packed[3]
            ms4, b4 = packed[4]
            cfg = kv.make_config(n_q, n_kv, B, w.iters, synth.sign_bits(w.seed))
            ws = kv.alloc_workspace(cfg, batch, max_blocks, dev)
            kvp = torch.empty(n_phys, n_kv, 2, B, D, dtype=torch.bfloat16, device=dev)
            kvp.normal_(generator=g)
            b16 = float((lens * n_kv * 512).sum() + batch * n_q * 768 + nbs.sum() * 4)
            ms16 = _time_events(lambda: kv.decode_attn_bf16(cfg, q, kvp, bt, sl, out, ws), reps, flush)
            assert kv.read_error(ws) == 0
            del kvp
            torch.cuda.empty_cache()
            print(json.dumps({"sweep_point": w.name, "batch": batch, "ctx": ctx,
                              "mean_len": float(lens.mean()),
                              "timing": "CUDA events, median of launches each queued behind a 1 GiB L2-flushing write",
                              "2bit": {"us": round(ms2 * 1e3, 2), "GB_per_s": round(b2 / ms2 / 1e6, 1),
                                       "tokens_per_s": round(batch / ms2 * 1e3, 1), "bytes": int(b2)},
                              "3bit": {"us": round(ms3 * 1e3, 2), "GB_per_s": round(b3 / ms3 / 1e6, 1),
                                       "tokens_per_s": round(batch / ms3 * 1e3, 1), "bytes": int(b3)},
                              "4bit": {"us": round(ms4 * 1e3, 2), "GB_per_s": round(b4 / ms4 / 1e6, 1),
                                       "tokens_per_s": round(batch / ms4 * 1e3, 1), "bytes": int(b4)},
                              "bf16": {"us": round(ms16 * 1e3, 2), "GB_per_s": round(b16 / ms16 / 1e6, 1),
                                       "tokens_per_s": round(batch / ms16 * 1e3, 1), "bytes": int(b16)},
                              "speedup_2bit_vs_bf16": round(ms16 / ms2, 2),
                              "speedup_3bit_vs_bf16": round(ms16 / ms3, 2),
                              "speedup_4bit_vs_bf16": round(ms16 / ms4, 2)}), flush=True)


# ---------------------------------------------------------------------------- Llama-3.1-8B layer

def run_llama_layer(args):
    """The Llama-3.1-8B layer workload: 16 sequences cached to 4095 tokens
    (127 blocks of 32 in the pool, 31 rows in staging); one step = the append
    of token 4096 (which completes every open block and quantises it) and
    decode attention over the 128 blocks. The cache (61 MB) fits in L2, so
    every rep runs after a 1 GiB L2-flushing write; CUDA events around each
    call, median over the reps."""
    import numpy as np
    import torch
    import bit_kv_cache_08_gb300 as kv
    import synth
    kv.build()
    dev = "cuda"
    w = synth.LLAMA8B_LAYER
    B, n_kv, n_q, batch, L = w.block, w.n_kv, w.n_q, w.batch, w.ctx
    nb = L // B
    sb = synth.sign_bits(w.seed)
    cfg = kv.make_config(n_q, n_kv, B, w.iters, sb)
    g = synth.make_gen(w.seed, dev)
    perm = np.random.default_rng(w.seed).permutation(batch * nb).astype(np.int32)
    bt = torch.from_numpy(perm.reshape(batch, nb)).to(dev)
    pool = kv.alloc_pool(cfg, batch * nb, dev)
    staging = kv.alloc_staging(cfg, batch, dev)
    ws = kv.alloc_workspace(cfg, batch, nb, dev)
    hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
    new = []
    for kind in (0, 1):
        T = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, dev).to(torch.bfloat16)
        offs = (bt[:, None, :nb - 1].long() * bb + (2 * torch.arange(n_kv, device=dev)[None, :, None] + kind)
                * hb).reshape(-1).contiguous()
        kv.quantize_block(cfg, kind, T[:, :, :(nb - 1) * B].contiguous(), pool, ws, dst_offsets=offs,
                          n_head_blocks=offs.numel())
        staging[:, :, kind, :B - 1] = T[:, :, (nb - 1) * B:L - 1]
        new.append(T[:, :, L - 1].contiguous())
        del T
    q = synth.queries(g, batch, n_q, dev).to(torch.bfloat16)
    pos = torch.full((batch,), L - 1, dtype=torch.int32, device=dev)
    lens = torch.full((batch,), L, dtype=torch.int32, device=dev)
    out = torch.empty(batch, n_q, D, device=dev)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    reps = max(50, args.steps)
    app, att, stp = [], [], []
    for r in range(args.warmup + reps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        kv.append(cfg, pool, staging, bt, pos, new[0], new[1], ws)
        e[1].record()
        kv.decode_attn(cfg, q, pool, staging, bt, lens, out, ws)
        e[2].record()
        torch.cuda.synchronize()
        if r >= args.warmup:
            app.append(e[0].elapsed_time(e[1]))
            att.append(e[1].elapsed_time(e[2]))
            stp.append(e[0].elapsed_time(e[2]))
    assert kv.read_error(ws) == 0
    peak, peak_kind = measured_peaks()
    attn_bytes = batch * L * n_kv * (2 * (32 + 16 + 2) + 2 * 256 / B) + batch * n_q * (D * 2 + D * 4) + batch * nb * 4
    app_bytes = batch * n_kv * 2 * (D * 2 + (B - 1) * D * 2 + hb)
    ma, mt, ms = statistics.median(app), statistics.median(att), statistics.median(stp)
    with ClockSampler(torch.cuda.current_device()) as clk:   # clocks over a second pass of the same reps
        for _ in range(reps):
            flush.zero_()
            kv.append(cfg, pool, staging, bt, pos, new[0], new[1], ws)
            kv.decode_attn(cfg, q, pool, staging, bt, lens, out, ws)
        torch.cuda.synchronize()
    print(json.dumps({
        "workload": w.name, "batch": batch, "seq_len": L, "n_q_heads": n_q, "n_kv_heads": n_kv, "block": B,
        "varn_iters": w.iters, "reps": reps,
        "timing": "CUDA events on the launching stream, median of reps each after a 1 GiB L2-flushing write",
        "append": {"us": round(ma * 1e3, 2), "algorithmic_bytes": int(app_bytes),
                   "GB_per_s": round(app_bytes / ma / 1e6, 1),
                   "head_blocks_quantised": batch * n_kv * 2,
                   "rows_per_s": round(batch * n_kv * 2 / (ma * 1e-3), 1)},
        "decode_attn": {"us": round(mt * 1e3, 2), "algorithmic_bytes": int(attn_bytes),
                        "GB_per_s": round(attn_bytes / mt / 1e6, 1),
                        "frac_of_hbm_peak": round(attn_bytes / mt / 1e6 / peak, 4), "peak": peak,
                        "peak_source": f"{peak_kind} HBM copy bandwidth"},
        "step": {"us": round(ms * 1e3, 2), "decode_tokens_per_s": round(batch / (ms * 1e-3), 1)},
        "roofline_time_us_at_100_70_pct": [round(attn_bytes / peak / 1e3, 2),
                                           round(attn_bytes / peak / 1e3 / 0.7, 2)],
        "clocks": clk.summary()}), flush=True)


# ---------------------------------------------------------------------------- Phi-4 long horizon

LONG_CHECK = (1, 64, 1024, 4096, 16384)


def run_long(args):
    """The Phi-4-14B long-horizon pseudo-decode: 40 layers, 40 query / 10 kv
    heads, batch 8 with prefill lengths uniform in [1024, 2048], then
    --long-steps steps, each appending one token per sequence to every layer
    and running decode attention on it. The first window of steps runs as
    eager C-ABI calls; after it the whole step (one gather of the step's new
    tokens for every layer, then every layer's kvarn_append and
    kvarn_decode_attn, then the position counters) is captured once as a
    CUDA graph and replayed, the serving loop's form: the entry points only
    enqueue kernels with fixed grids, and lengths and positions live in
    device tensors. CUDA events per window of steps. At the checkpoint steps, every layer's output is also
    computed over a bf16 cache holding the same tokens (the repo's bf16-cache
    kernel), and the 2-bit error against it is reported: max and mean of
    |o_2bit - o_bf16| / max(1, |o_bf16|) and the relative L2 norm over all
    layers, sequences and heads."""
    import numpy as np
    import torch
    import bit_kv_cache_08_gb300 as kv
    import synth
    kv.build()
    dev = "cuda"
    w = synth.PHI4_LONG
    B, n_kv, n_q, batch, layers = w.block, w.n_kv, w.n_q, w.batch, w.layers
    steps = args.long_steps
    prefill = synth.prefill_lengths(batch, 1024, 2048, w.seed)
    Lmax = max(prefill) + steps
    mb = (Lmax + B - 1) // B
    st = []
    # every layer's appended tokens: [K|V][layer][step][batch][n_kv][128]
    NEWS = torch.empty(2, layers, steps, batch, n_kv, D, dtype=torch.bfloat16, device=dev)
    t_setup = time.time()
    for l in range(layers):
        sb = synth.sign_bits(100 + l)
        cfg = kv.make_config(n_q, n_kv, B, w.iters, sb)
        g = synth.make_gen(w.seed * 100 + l, dev)
        perm = np.random.default_rng([w.seed, l]).permutation(batch * mb).astype(np.int32)
        bt = torch.from_numpy(perm.reshape(batch, mb)).to(dev)
        pool = kv.alloc_pool(cfg, batch * mb, dev)
        staging = kv.alloc_staging(cfg, batch, dev)
        ws = kv.alloc_workspace(cfg, batch, mb, dev)
        kvp = torch.zeros(batch * mb, n_kv, 2, B, D, dtype=torch.bfloat16, device=dev)   # bf16 pages
        hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
        steps_idx = torch.arange(steps, device=dev)[:, None] + torch.tensor(prefill, device=dev)[None, :]
        for kind in (0, 1):
            T = synth.kv_values(g, batch, n_kv, mb * B, w.sigma_m, w.n_out, w.out_factor, dev).to(torch.bfloat16)
            # every token in the bf16 pages (tokens past a sequence's length are never read)
            kvp[bt.reshape(-1).long(), :, kind] = T.view(batch, n_kv, mb, B, D).permute(0, 2, 1, 3, 4).reshape(
                batch * mb, n_kv, B, D)
            # the 2-bit cache: the prefill's full blocks quantised, its open tail in staging
            for b, Lb in enumerate(prefill):
                nbf = Lb // B
                offs = (bt[b, :nbf].long()[None, :] * bb + (2 * torch.arange(n_kv, device=dev)[:, None] + kind)
                        * hb).reshape(-1).contiguous()
                kv.quantize_block(cfg, kind, T[b, :, :nbf * B].contiguous(), pool, ws, dst_offsets=offs,
                                  n_head_blocks=offs.numel())
                staging[b, :, kind, :Lb - nbf * B] = T[b, :, nbf * B:Lb]
            # the appended tokens of every step: [steps][batch][n_kv][128]
            NEWS[kind, l] = T[torch.arange(batch, device=dev)[None, :], :, steps_idx]
            del T
        q = synth.queries(g, batch, n_q, dev).to(torch.bfloat16)
        st.append(dict(cfg=cfg, bt=bt, pool=pool, staging=staging, ws=ws, kvp=kvp, q=q,
                       out=torch.empty(batch, n_q, D, device=dev)))
        torch.cuda.synchronize()
        assert kv.read_error(ws) == 0
    t_setup = time.time() - t_setup
    pos = torch.tensor(prefill, dtype=torch.int32, device=dev)
    lens = pos + 1
    ws16 = kv.alloc_workspace(st[0]["cfg"], batch, mb, dev)
    ref = torch.empty(batch, n_q, D, device=dev)
    window = 256
    windows, curve = [], []
    win_ms, win_n = 0.0, 0

    def mark():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    # the step's new tokens for every layer, gathered into fixed buffers
    sidx = torch.zeros(1, dtype=torch.long, device=dev)
    buf = torch.empty(2, layers, 1, batch, n_kv, D, dtype=torch.bfloat16, device=dev)

    kbuf = [buf[0, l, 0] for l in range(layers)]
    vbuf = [buf[1, l, 0] for l in range(layers)]
    torch.index_select(NEWS, 2, sidx, out=buf)   # loads the gather's kernel before the timed windows
    torch.cuda.synchronize()

    def one_step():
        torch.index_select(NEWS, 2, sidx, out=buf)
        for l, x in enumerate(st):
            kv.append(x["cfg"], x["pool"], x["staging"], x["bt"], pos, kbuf[l], vbuf[l], x["ws"])
            kv.decode_attn(x["cfg"], x["q"], x["pool"], x["staging"], x["bt"], lens, x["out"], x["ws"])
        pos.add_(1)
        lens.add_(1)
        sidx.add_(1)

    eager_steps = min(window, steps)   # the first window runs eagerly
    graph = None
    ev0 = mark()
    t_loop = time.time()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for s in range(1, steps + 1):
            if graph is None:
                one_step()
            else:
                graph.replay()
            win_n += 1
            check = s in LONG_CHECK or s == steps
            if check or s % window == 0 or s == steps:
                ev1 = mark()
                torch.cuda.synchronize()
                win_ms += ev0.elapsed_time(ev1)
                if s % window == 0 or s == steps:
                    windows.append((s, win_ms * 1e3 / win_n))
                    win_ms, win_n = 0.0, 0
                if s == eager_steps and s < steps and not args.long_eager:   # capture once, outside the timed windows
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph):
                        one_step()
                if check:      # outside the timed windows
                    num = den = 0.0
                    emax = emean = 0.0
                    for x in st:
                        kv.decode_attn_bf16(x["cfg"], x["q"], x["kvp"], x["bt"], lens, ref, ws16)
                        d = (x["out"] - ref).abs() / ref.abs().clamp_min(1.0)
                        emax = max(emax, float(d.max()))
                        emean += float(d.mean()) / layers
                        num += float(((x["out"] - ref) ** 2).sum())
                        den += float((ref ** 2).sum())
                    curve.append({"step": s, "tokens_min": int(lens.min()), "tokens_max": int(lens.max()),
                                  "max_rel": round(emax, 5), "mean_rel": round(emean, 6),
                                  "rel_l2": round(math.sqrt(num / den), 6)})
                ev0 = mark()
    t_loop = time.time() - t_loop
    for x in st:
        assert kv.read_error(x["ws"]) == 0
    assert kv.read_error(ws16) == 0
    us = [u for _, u in windows]
    ug = us[1:] if len(us) > 1 else us   # the graph-replayed windows (eager with --long-eager)
    print(json.dumps({
        "workload": w.name, "layers": layers, "batch": batch, "n_q_heads": n_q, "n_kv_heads": n_kv, "block": B,
        "varn_iters": w.iters, "prefill_lengths": prefill, "steps": steps,
        "timing": f"CUDA events per window of {window} steps (each step: one gather of the step's new tokens, "
                  "then for every layer kvarn_append + kvarn_decode_attn); the first window as eager calls, the "
                  "rest as replays of the step captured once as a CUDA graph; the error checkpoints and the "
                  "capture are outside the windows",
        "us_per_step": {"first_window_eager": round(us[0], 1),
                        "second_window_graph": round(us[1], 1) if len(us) > 1 else None,
                        "last_window": round(us[-1], 1),
                        "mean_graph": round(sum(ug) / len(ug), 1),
                        "by_step": [[s_, round(u, 1)] for s_, u in windows[::max(1, len(windows) // 16)]]},
        "decode_tokens_per_s_mean": round(batch / (sum(ug) / len(ug) * 1e-6), 1),
        "error_vs_bf16_cache": curve, "setup_s": round(t_setup, 1), "loop_s": round(t_loop, 1),
        "clocks": clk.summary()}), flush=True)


# ---------------------------------------------------------------------------- chunked prefill

PREFILL_CHUNKS = (1, 4, 16, 64)


def run_prefill(args):
    """kvarn_prefill_attn on the Llama-3.1-8B layer: every sequence holds 4096
    tokens, the last `chunk` of them are the chunk's queries. Each launch is
    timed alone after a 1 GiB L2-flushing write (median). Reported: query rows
    per second and the cache bytes of one pass over the visible cache per
    launch, divided by its time (every row re-reads its prefix; the repeats
    come from L2)."""
    import torch
    import bit_kv_cache_08_gb300 as kv
    import synth
    kv.build()
    dev = "cuda"
    w = synth.LLAMA8B_LAYER
    B, n_kv, n_q, batch, L = w.block, w.n_kv, w.n_q, w.batch, w.ctx
    nb = L // B
    sb = synth.sign_bits(w.seed)
    cfg = kv.make_config(n_q, n_kv, B, w.iters, sb)
    g = synth.make_gen(w.seed, dev)
    bt = torch.arange(batch * nb, dtype=torch.int32, device=dev).view(batch, nb)
    pool = kv.alloc_pool(cfg, batch * nb, dev)
    staging = kv.alloc_staging(cfg, batch, dev)
    ws0 = kv.alloc_workspace(cfg, 0, 0, dev)
    hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
    for kind in (0, 1):
        T = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, dev).to(torch.bfloat16)
        offs = (bt[:, None, :].long() * bb + (2 * torch.arange(n_kv, device=dev)[None, :, None] + kind) * hb)
        kv.quantize_block(cfg, kind, T.contiguous(), pool, ws0, dst_offsets=offs.reshape(-1).contiguous(),
                          n_head_blocks=batch * n_kv * nb)
        del T
    lens = torch.full((batch,), L, dtype=torch.int32, device=dev)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    cache_bytes = batch * nb * bb            # every (kv head, K, V) head-block once
    for chunk in PREFILL_CHUNKS:
        q = synth.queries(g, batch * chunk, n_q, dev).reshape(batch, chunk, n_q, D).to(torch.bfloat16)
        out = torch.empty(batch, chunk, n_q, D, device=dev)
        ws = kv.alloc_prefill_workspace(cfg, batch, chunk, nb, dev)
        for _ in range(3):
            kv.prefill_attn(cfg, q, pool, staging, bt, lens, out, ws)
        ms = _time_events(lambda: kv.prefill_attn(cfg, q, pool, staging, bt, lens, out, ws), 10, flush)
        assert kv.read_error(ws) == 0
        print(json.dumps({"prefill_chunk": chunk, "workload": w.name, "batch": batch, "cached_tokens": L,
                          "us": round(ms * 1e3, 1), "query_rows_per_s": round(batch * chunk / ms * 1e3, 1),
                          "cache_GB_per_s_one_pass": round(cache_bytes / ms / 1e6, 1),
                          "timing": "CUDA events, median of 10 launches each after a 1 GiB L2-flushing write"}),
              flush=True)
        del q, out, ws


# ---------------------------------------------------------------------------- ablation

ABLATIONS = (  # (name, flags, iters, bits): the pages' ablation list, plus the two ends and 4-bit codes
    ("kvarn (full)", 0, 3, 2),
    ("hadamard only", 0, 0, 2),
    ("varn only (no rotation)", 1, 3, 2),
    ("varn token axis only", 4, 3, 2),
    ("varn channel axis only", 2, 3, 2),
    ("plain group 2-bit", 1, 0, 2),
    ("kvarn 3-bit", 0, 3, 3),
    ("kvarn 4-bit", 0, 3, 4),
    ("plain group 4-bit", 1, 0, 4),
)


def run_ablation(args):
    """Attention-output and reconstruction error of each ablation against the
    bf16 cache holding the same tokens, on the Llama-3.1-8B layer workload
    (batch 16, 4096 tokens, block 32), one JSON line per variant."""
    import numpy as np
    import torch
    import bit_kv_cache_08_gb300 as kv
    import synth
    kv.build()
    dev = "cuda"
    w = synth.LLAMA8B_LAYER
    B, n_kv, n_q, batch, L = w.block, w.n_kv, w.n_q, w.batch, w.ctx
    nb = L // B
    g = synth.make_gen(w.seed, dev)
    K = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, dev).to(torch.bfloat16)
    V = synth.kv_values(g, batch, n_kv, L, w.sigma_m, w.n_out, w.out_factor, dev).to(torch.bfloat16)
    q = synth.queries(g, batch, n_q, dev).to(torch.bfloat16)
    bt = torch.arange(batch * nb, dtype=torch.int32, device=dev).view(batch, nb)
    lens = torch.full((batch,), L, dtype=torch.int32, device=dev)
    sb = synth.sign_bits(w.seed)
    # the bf16 reference: same tokens, plain pages
    kvp = torch.stack([K.view(batch, n_kv, nb, B, D), V.view(batch, n_kv, nb, B, D)], dim=3)   # [b][h][j][2][B][D]
    kvp = kvp.permute(0, 2, 1, 3, 4, 5).reshape(batch * nb, n_kv, 2, B, D).contiguous()
    cfg0 = kv.make_config(n_q, n_kv, B, 3, sb)
    ref = torch.empty(batch, n_q, D, device=dev)
    kv.decode_attn_bf16(cfg0, q, kvp, bt, lens, ref, kv.alloc_workspace(cfg0, batch, nb, dev))
    del kvp
    for name, flags, iters, bits in ABLATIONS:
        cfg = kv.make_config(n_q, n_kv, B, iters, sb, flags=flags, bits=bits)
        pool = kv.alloc_pool(cfg, batch * nb, dev)
        staging = kv.alloc_staging(cfg, batch, dev)
        ws = kv.alloc_workspace(cfg, batch, nb, dev)
        hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
        rec, split = [], []
        for kind, T in ((0, K), (1, V)):
            offs = (bt[:, None, :].long() * bb + (2 * torch.arange(n_kv, device=dev)[None, :, None] + kind) * hb)
            kv.quantize_block(cfg, kind, T.contiguous(), pool, ws, dst_offsets=offs.reshape(-1).contiguous(),
                              n_head_blocks=batch * n_kv * nb)
            deq = torch.empty(batch * n_kv * nb, B, D, device=dev)
            kv.dequantize(cfg, kind, pool, deq, rotated=False, src_offsets=offs.reshape(-1).contiguous())
            x = T.float().reshape(-1, B, D)
            rec.append(float(((deq - x) ** 2).sum() / (x ** 2).sum()))
            es = torch.empty(batch * n_kv * nb, B, 4, device=dev)
            kv.error_decomposition(cfg, kind, T.contiguous(), pool, es, packed_offsets=offs.reshape(-1).contiguous(),
                                   n_head_blocks=batch * n_kv * nb)
            es = es.reshape(-1, 4)
            top = es[:, 0] >= torch.quantile(es[:, 0], 0.9)
            split.append({"em_over_ed_energy": round(float((es[:, 2] ** 2).sum() / (es[:, 3] ** 2).sum()), 4),
                          "em_dominant_frac": round(float((es[:, 2] > es[:, 3]).float().mean()), 4),
                          "em_dominant_frac_top_norm_decile": round(float((es[top, 2] > es[top, 3]).float().mean()), 4)})
        out = torch.empty(batch, n_q, D, device=dev)
        kv.decode_attn(cfg, q, pool, staging, bt, lens, out, ws)
        torch.cuda.synchronize()
        assert kv.read_error(ws) == 0
        d = out - ref
        cos = torch.nn.functional.cosine_similarity(out.reshape(-1, D), ref.reshape(-1, D), dim=1)
        print(json.dumps({"ablation": name, "flags": flags, "varn_iters": iters, "bits": bits, "workload": w.name,
                          "attn_rel_l2_vs_bf16": round(float(d.norm() / ref.norm()), 5),
                          "attn_mean_cosine_vs_bf16": round(float(cos.mean()), 5),
                          "k_rel_mse": round(rec[0], 5), "v_rel_mse": round(rec[1], 5),
                          "error_split_k": split[0], "error_split_v": split[1]}), flush=True)
        del pool, staging, ws
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.llama_layer:
        run_llama_layer(args)
        return
    if args.long:
        run_long(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.ablation:
        run_ablation(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        tdist.init_process_group("nccl")
        if rank == 0:                      # one in-tree build, the other ranks then load it
            from bit_kv_cache_08_gb300.build import build as build_lib
            build_lib()
        tdist.barrier()
    res, state, objs = run_gpu(args, rank, world)
    w = workload()
    res["e2e"] = e2e_gpu(args, objs, state, w, world)
    import torch
    if rank == 0 and not args.no_bf16:
        del state
        torch.cuda.empty_cache()
        res["bf16_cache_comparison"] = bf16_comparison(objs[0], w, torch.cuda.current_device())
        res["quantize_bulk"] = bulk_quantize(objs[0], w, torch.cuda.current_device(), res["roofline"]["peak"])
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
