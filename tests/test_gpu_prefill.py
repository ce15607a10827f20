"""Chunked prefill attention on the GPU (each chunk row causal over the
packed cache as it stands) against the fp64 oracle over the same bytes."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from kvtest_util import PagedCache, attn_close, bf16_bits

pytestmark = pytest.mark.gpu
D = 128


def _prefill(kv, cache, q, lens, split=True):
    """split: the workspace sized for the full block split (else the minimum)."""
    cfg = cache.cfg
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.full(q.shape, float("nan"), device="cuda")
    ws = (kv.alloc_prefill_workspace(cfg, q.shape[0], q.shape[1], cache.max_blocks) if split
          else kv.alloc_workspace(cfg, q.shape[0] * q.shape[1], cache.max_blocks))
    kv.prefill_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), kv.read_error(ws)


def _oracle(cache, q, lens, sb, sm_scale=None):
    cfg = cache.cfg
    sm_scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    return oracle.prefill_attention(cfg.block_size, cfg.n_q_heads, cfg.n_kv_heads, sb, sm_scale,
                                    q.double().cpu().numpy(), cache.pool.cpu().numpy(), bf16_bits(cache.staging),
                                    cache.block_table_np, np.asarray(lens, np.int32), flags=int(cfg.flags),
                                    bits=int(cfg.bits))


def _cache(kv, B, bits, iters, n_q, n_kv, lens, seed):
    sb = synth.sign_bits(seed)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb, bits=bits)
    g = synth.make_gen(seed)
    Lmax = max(lens)
    K = synth.kv_values(g, len(lens), n_kv, Lmax, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, len(lens), n_kv, Lmax, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, len(lens), (Lmax + B - 1) // B + 1, perm_seed=seed)
    cache.prefill(K, V, lens)
    return cache, sb, g


@pytest.mark.parametrize("B,bits,iters", [(32, 2, 3), (64, 2, 2), (32, 3, 3), (64, 3, 2), (32, 4, 3), (64, 4, 2)])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float32])
def test_prefill_ragged_chunks_match_oracle(kvlib, B, bits, iters, qdtype):
    """A 40-row chunk over ragged sequences: rows inside complete blocks (the
    causal cut inside a quantised block), rows in the raw tail, a sequence
    shorter than the chunk (rows at negative positions give zeros) and one
    exactly as long as the chunk."""
    kv = kvlib
    n_q, n_kv, chunk = 8, 2, 40
    lens = [3 * B + 7, 2 * B, 25, 40, 700]
    cache, sb, g = _cache(kv, B, bits, iters, n_q, n_kv, lens, 40 + B + bits)
    q = synth.queries(g, len(lens) * chunk, n_q).reshape(len(lens), chunk, n_q, D).to(qdtype).cuda()
    got, err = _prefill(kv, cache, q, lens)
    assert err == 0
    ref = _oracle(cache, q, lens, sb)
    assert np.all(got[2, :chunk - 25] == 0.0)         # positions < 0
    attn_close(got, ref)


def test_prefill_chunk_of_one_matches_decode(kvlib):
    kv = kvlib
    B, n_q, n_kv = 64, 32, 8
    lens = [1000, 64, 1, 333]
    cache, sb, g = _cache(kv, B, 2, 2, n_q, n_kv, lens, 77)
    q = synth.queries(g, len(lens), n_q).to(torch.bfloat16).cuda()
    pre, err = _prefill(kv, cache, q[:, None].contiguous(), lens)
    assert err == 0
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    dec = torch.empty(len(lens), n_q, D, device="cuda")
    ws = kv.alloc_workspace(cache.cfg, len(lens), cache.max_blocks)
    kv.decode_attn(cache.cfg, q, cache.pool, cache.staging, cache.block_table, sl, dec, ws)
    torch.cuda.synchronize()
    d = dec.cpu().double().numpy()
    np.testing.assert_allclose(pre[:, 0], d, rtol=1e-5, atol=1e-5)
    ref = _oracle(cache, q[:, None], lens, sb)
    attn_close(pre, ref)


@pytest.mark.parametrize("G", [1, 2, 3])
def test_prefill_long_chunk_many_partials(kvlib, G):
    """2048-token sequences, a 96-row chunk: every row is split over several
    warps and merged, with the causal cut in the last visible block."""
    kv = kvlib
    B, n_kv = 32, 2
    lens = [2048, 1500]
    cache, sb, g = _cache(kv, B, 2, 3, G * n_kv, n_kv, lens, 90 + G)
    chunk = 96
    q = synth.queries(g, len(lens) * chunk, G * n_kv).reshape(len(lens), chunk, G * n_kv, D).to(
        torch.bfloat16).cuda()
    got, err = _prefill(kv, cache, q, lens)
    assert err == 0
    attn_close(got, _oracle(cache, q, lens, sb))


def test_prefill_minimum_workspace_gives_the_same_rows(kvlib):
    """The block split adapts to the workspace passed: the minimum workspace
    (fewer splits) gives the same rows up to rounding."""
    kv = kvlib
    B, n_q, n_kv = 32, 8, 2
    lens = [900, 333]
    cache, sb, g = _cache(kv, B, 2, 3, n_q, n_kv, lens, 61)
    q = synth.queries(g, len(lens) * 6, n_q).reshape(len(lens), 6, n_q, D).to(torch.bfloat16).cuda()
    a, err_a = _prefill(kv, cache, q, lens, split=True)
    b, err_b = _prefill(kv, cache, q, lens, split=False)
    assert err_a == 0 and err_b == 0
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5)
    attn_close(b, _oracle(cache, q, lens, sb))


def test_prefill_bad_length_is_flagged(kvlib):
    kv = kvlib
    B = 32
    cache, sb, g = _cache(kv, B, 2, 3, 4, 1, [64], 5)
    q = synth.queries(g, 4, 4).reshape(1, 4, 4, D).cuda()
    got, err = _prefill(kv, cache, q, [cache.max_blocks * B + 1])
    assert err & kv.DEVERR_POSITION


@pytest.mark.parametrize("flags,iters", [(oracle.NO_ROTATION, 3), (0, 0), (oracle.NO_TOKEN_PASS, 2)])
def test_prefill_with_ablation_switches(kvlib, flags, iters):
    """A cache written with an ablation switch is read with it: no rotation
    (queries and output stay unrotated), Hadamard only, one VarN axis."""
    kv = kvlib
    B, n_q, n_kv = 32, 8, 2
    lens = [300, 77]
    sb = synth.sign_bits(70 + flags)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb, flags=flags)
    g = synth.make_gen(71 + flags)
    K = synth.kv_values(g, len(lens), n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, len(lens), n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, len(lens), (max(lens) + B - 1) // B + 1, perm_seed=flags)
    cache.prefill(K, V, lens)
    q = synth.queries(g, len(lens) * 12, n_q).reshape(len(lens), 12, n_q, D).cuda()
    got, err = _prefill(kv, cache, q, lens)
    assert err == 0
    attn_close(got, _oracle(cache, q, lens, sb))
