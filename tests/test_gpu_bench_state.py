"""The benchmark's own state after its timed graph replays: bench.py's
Qwen3-4B-shaped step (two of its layers, the same prefill, tables and
inputs), captured once as a CUDA graph and replayed the way the timed region
replays it; then sampled (layer, sequence) outputs are checked against the
oracle over the cache bytes the replays left behind, and the block every
step re-completes against the oracle's staged quantisation."""
import math
from collections import Counter

import numpy as np
import pytest
import torch

import bench
import oracle
from kvtest_util import assert_code_flip_rate, attn_close, bf16_bits, staged_quantize_parity

pytestmark = pytest.mark.gpu
D = 128


def test_bench_state_after_graph_replays(kvlib):
    kv = kvlib
    w = bench.workload()
    layers, replays = 2, 3
    state = bench.build_layers(kv, w, layers, "cuda")
    B, batch, nb = w.block, w.batch, w.ctx // w.block
    ws = kv.alloc_workspace(state[0]["cfg"], batch, nb, "cuda")
    pos = torch.full((batch,), w.ctx - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((batch,), w.ctx, dtype=torch.int32, device="cuda")
    out = torch.full((layers, batch, w.n_q, D), float("nan"), device="cuda")

    def step():
        for l, st in enumerate(state):
            kv.append(st["cfg"], st["pool"], st["staging"], st["bt"], pos, st["k_new"], st["v_new"], ws)
            kv.decode_attn(st["cfg"], st["q"], st["pool"], st["staging"], st["bt"], lens, out[l], ws)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.fill_(float("nan"))
    for _ in range(replays):
        graph.replay()
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    got = out.cpu().double().numpy()
    assert np.all(np.isfinite(got))

    for l, seqs in ((0, [0, 63]), (1, [37])):
        st = state[l]
        cfg = st["cfg"]
        sb = [int(x) for x in cfg.sign_bits]
        pool_np = st["pool"].cpu().numpy()
        bt = st["bt"].cpu().numpy()
        ref = oracle.decode_attention(B, w.n_q, w.n_kv, sb, 1.0 / math.sqrt(D),
                                      st["q"][seqs].double().cpu().numpy(), pool_np,
                                      bf16_bits(st["staging"][seqs]), np.ascontiguousarray(bt[seqs]),
                                      np.full(len(seqs), w.ctx, dtype=np.int32))
        attn_close(got[l][seqs], ref)

        # the last block of sequence seqs[0], kv head 5, re-completed by every step:
        # its 63 staged rows plus the appended one, against the oracle's quantisation
        b, h, j = seqs[0], 5, nb - 1
        hb, bb = kv.head_block_bytes(cfg), kv.block_bytes(cfg)
        total = Counter()
        for kind, new in ((0, st["k_new"]), (1, st["v_new"])):
            rows = torch.cat([st["staging"][b, h, kind, :B - 1].float(), new[b, h][None].float()]).double()
            o = int(bt[b, j]) * bb + (2 * h + kind) * hb
            got_block = pool_np.reshape(-1)[o:o + hb]
            total.update(staged_quantize_parity(rows.cpu().numpy()[None], got_block[None], B, w.iters, kind, sb))
        assert_code_flip_rate(total)
