"""The long-horizon pseudo-decode workload (Phi-4-14B shape) and the ragged
throughput-sweep shapes (Llama-3.1-8B layer), on the GPU, checked against the
oracle over the GPU's own cache bytes at sampled steps / sequences.

The long-horizon test also tracks, at every step, the attention-output
difference between the 2-bit cache and a bf16 cache holding the same tokens
(the synthetic stand-in for the pages' error-versus-decode-step curves; the
outputs do not feed back, so growth here comes only from the growing cache).
"""
import numpy as np
import pytest
import torch

import synth
from kvtest_util import PagedCache, attn_close, oracle_attention

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("layer", [0, 39])
def test_phi4_long_horizon_pseudo_decode(kvlib, layer):
    kv = kvlib
    w = synth.PHI4_LONG
    B, n_q, n_kv, batch = w.block, w.n_q, w.n_kv, w.batch
    steps = 16384                # the workload's appends, each followed by attention
    check_at = {1, 64, 1024, 4096, steps}
    prefill = synth.prefill_lengths(batch, 1024, 2048, w.seed)
    Lmax = max(prefill) + steps
    max_blocks = (Lmax + B - 1) // B
    sb = synth.sign_bits(100 + layer)
    cfg = kv.make_config(n_q, n_kv, B, w.iters, sb)
    g = synth.make_gen(w.seed * 100 + layer, "cuda")
    K = synth.kv_values(g, batch, n_kv, Lmax, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
    V = synth.kv_values(g, batch, n_kv, Lmax, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=layer)
    cache.prefill(K, V, prefill)
    # the bf16 comparison cache: the same tokens under the same block table, plain pages
    kvp = torch.zeros(batch * max_blocks, n_kv, 2, B, D, dtype=torch.bfloat16, device="cuda")
    for b in range(batch):
        for j in range(max_blocks):
            lo, hi = j * B, min((j + 1) * B, Lmax)
            kvp[cache.block_table_np[b, j], :, 0, :hi - lo] = K[b, :, lo:hi]
            kvp[cache.block_table_np[b, j], :, 1, :hi - lo] = V[b, :, lo:hi]
    ws = kv.alloc_workspace(cfg, batch, max_blocks)
    ws_bf = kv.alloc_workspace(cfg, batch, max_blocks)
    pos = torch.tensor(prefill, dtype=torch.int32, device="cuda")
    ar = torch.arange(batch, device="cuda")
    out = torch.empty(batch, n_q, D, device="cuda")
    ref16 = torch.empty(batch, n_q, D, device="cuda")
    curve = []
    for s in range(1, steps + 1):
        kv.append(cfg, cache.pool, cache.staging, cache.block_table, pos, K[ar, :, pos.long()].contiguous(),
                  V[ar, :, pos.long()].contiguous(), ws)
        pos += 1
        q = synth.queries(g, batch, n_q, "cuda").to(torch.bfloat16)
        kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, pos, out, ws)
        kv.decode_attn_bf16(cfg, q, kvp, cache.block_table, pos, ref16, ws_bf)
        d = (out - ref16).abs() / ref16.abs().clamp_min(1.0)
        curve.append(torch.stack([d.max(), d.mean()]))
        if s in check_at:
            torch.cuda.synchronize()
            assert kv.read_error(ws) == 0 and kv.read_error(ws_bf) == 0
            seqs = [0, batch - 1]
            ref = oracle_attention(cache, q, pos.cpu().numpy(), sb, seqs=seqs)
            attn_close(out.cpu().double().numpy()[seqs], ref)
    curve = torch.stack(curve).cpu().numpy()
    assert np.all(np.isfinite(curve))
    print(f"layer {layer}: 2-bit vs bf16 relative output difference (max, mean) at step 1 "
          f"{curve[0]}, 1024 {curve[1023]}, 4096 {curve[4095]}, {steps} {curve[-1]}")


@pytest.mark.parametrize("batch,ctx", [(1, 131072), (8, 32768), (256, 1024), (128, 8192), (32, 131072), (256, 32768),
                                       (128, 32768), (256, 131072)])
def test_llama_sweep_point(kvlib, batch, ctx):
    kv = kvlib
    w = synth.sweep_point(batch, ctx)
    B = w.block
    lens = w.seq_lens
    max_blocks = (max(lens) + B - 1) // B
    sb = synth.sign_bits(w.seed)
    cfg = kv.make_config(w.n_q, w.n_kv, B, w.iters, sb)
    g = synth.make_gen(w.seed + batch + ctx, "cuda")
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=batch)
    Lm = max(lens)
    # fill 16 sequences at a time to bound the raw K/V held on the device
    for b0 in range(0, batch, 16):
        bs = list(range(b0, min(batch, b0 + 16)))
        Kb = synth.kv_values(g, len(bs), w.n_kv, Lm, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
        Vb = synth.kv_values(g, len(bs), w.n_kv, Lm, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
        sub = PagedCache.__new__(PagedCache)
        sub.__dict__.update(cache.__dict__)
        sub.block_table_np = cache.block_table_np[bs]
        sub.staging = cache.staging[bs[0]:bs[-1] + 1]
        sub.prefill(Kb, Vb, [lens[b] for b in bs])
        del Kb, Vb
    q = synth.queries(g, batch, w.n_q, "cuda").to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.empty(batch, w.n_q, D, device="cuda")
    ws = kv.alloc_workspace(cfg, batch, max_blocks)
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    seqs = sorted({0, batch // 2, batch - 1})
    ref = oracle_attention(cache, q, lens, sb, seqs=seqs)
    attn_close(out.cpu().double().numpy()[seqs], ref)
