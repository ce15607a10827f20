"""The named workloads at full size on the GPU, in the launch configuration
bench.py times: the append that completes every open block, then one decode
attention, checked against the oracle over the same cache bytes (every output
for the Llama-8B layer; sampled sequences for the Qwen3-4B layer)."""
import numpy as np
import pytest
import torch

import synth
from collections import Counter

from kvtest_util import PagedCache, assert_code_flip_rate, attn_close, oracle_attention, staged_quantize_parity

pytestmark = pytest.mark.gpu


def _layer(kv, w, seed_extra=0, perm=True, bits=2):
    sb = synth.sign_bits(w.seed)
    cfg = kv.make_config(w.n_q, w.n_kv, w.block, w.iters, sb, bits=bits)
    g = synth.make_gen(w.seed + seed_extra, "cuda")
    K = synth.kv_values(g, w.batch, w.n_kv, w.ctx, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
    V = synth.kv_values(g, w.batch, w.n_kv, w.ctx, w.sigma_m, w.n_out, w.out_factor, "cuda").to(torch.bfloat16)
    q = synth.queries(g, w.batch, w.n_q, "cuda").to(torch.bfloat16)
    cache = PagedCache(kv, cfg, w.batch, w.ctx // w.block, perm_seed=(w.seed if perm else None))
    cache.prefill(K, V, [w.ctx - 1] * w.batch)
    ws = kv.alloc_workspace(cfg, w.batch, w.ctx // w.block)
    pos = torch.full((w.batch,), w.ctx - 1, dtype=torch.int32, device="cuda")
    kv.append(cfg, cache.pool, cache.staging, cache.block_table, pos, K[:, :, -1].contiguous(),
              V[:, :, -1].contiguous(), ws)
    lens = torch.full((w.batch,), w.ctx, dtype=torch.int32, device="cuda")
    out = torch.empty(w.batch, w.n_q, 128, device="cuda")
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, lens, out, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    return sb, cfg, K, V, q, cache, out.cpu().double().numpy()


def _check_appended(w, sb, K, V, cache, samples, bits=2):
    B = w.block
    j = w.ctx // B - 1
    total = Counter()
    for (b, h) in samples:
        for kind, T in ((0, K), (1, V)):
            rows = T[b, h, j * B:(j + 1) * B].double().cpu().numpy()
            total.update(staged_quantize_parity(rows[None], cache.head_block(b, h, j, kind)[None], B, w.iters,
                                                kind, sb, bits=bits))
    assert_code_flip_rate(total)


def test_llama8b_layer(kvlib):
    w = synth.LLAMA8B_LAYER
    sb, cfg, K, V, q, cache, got = _layer(kvlib, w)
    _check_appended(w, sb, K, V, cache, [(0, 0), (5, 3), (15, 7)])
    ref = oracle_attention(cache, q, [w.ctx] * w.batch, sb)
    worst = attn_close(got, ref)
    print("llama8b layer worst error ratio", worst)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_qwen3_4b_layer_sampled(kvlib, bits):
    """The 36-layer workload's layer shape at full size (64 x 8192 tokens,
    B = 64), at every code width."""
    w = synth.QWEN3_4B_CACHE
    sb, cfg, K, V, q, cache, got = _layer(kvlib, w, bits=bits)
    _check_appended(w, sb, K, V, cache, [(0, 0), (63, 7)], bits=bits)
    seqs = [0, 21, 63]
    ref = oracle_attention(cache, q, [w.ctx] * w.batch, sb, seqs=seqs)
    worst = attn_close(got[seqs], ref)
    print(f"qwen3-4b layer {bits}-bit (sampled) worst error ratio", worst)
