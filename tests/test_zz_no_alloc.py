"""kvarn_decode_attn_noalloc: the decode-attention entry point that allocates
nothing (its scratch is compiled into the library), for callers that can
only pass inputs and outputs. Called through the C ABI twice in a row, each
result must match kvarn_decode_attn on the same cache, and the fp64 oracle
over the same cache bytes, within the attention tolerance the other tests
use; at both block sizes and at 2- and 4-bit codes. Kept in the file pytest
collects last."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from kvtest_util import PagedCache, attn_close, oracle_attention

pytestmark = pytest.mark.gpu
D = 128


def _noalloc(kv, cfg, q, cache, lens, out, err):
    return kv.lib().kvarn_decode_attn_noalloc(
        ctypes.byref(cfg), ctypes.c_void_p(q.data_ptr()), 0 if q.dtype == torch.bfloat16 else 1,
        ctypes.c_void_p(cache.pool.data_ptr()), cache.pool.shape[0], ctypes.c_void_p(cache.staging.data_ptr()),
        ctypes.c_void_p(cache.block_table.data_ptr()), cache.block_table.shape[1],
        ctypes.c_void_p(lens.data_ptr()), q.shape[0], ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("B,bits", [(32, 2), (64, 2), (32, 4), (64, 4)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(kvlib, B, bits):
    kv = kvlib
    n_q, n_kv = 8, 2
    lens_list = [5 * B + 7, 3 * B, 1, 700]
    batch = len(lens_list)
    sb = synth.sign_bits(31)
    cfg = kv.make_config(n_q, n_kv, B, 3, sb, bits=bits)
    g = synth.make_gen(31)
    K = synth.kv_values(g, batch, n_kv, max(lens_list), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens_list), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, (max(lens_list) + B - 1) // B, perm_seed=31)
    cache.prefill(K, V, lens_list)
    lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
    ws = kv.alloc_workspace(cfg, batch, cache.max_blocks)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        q = synth.queries(g, batch, n_q).to(torch.bfloat16).cuda()
        ref = torch.empty(batch, n_q, D, device="cuda")
        kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, lens, ref, ws)
        out = torch.full((batch, n_q, D), float("nan"), device="cuda")
        assert _noalloc(kv, cfg, q, cache, lens, out, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error flags {int(err.item())}"
        got = out.cpu().double().numpy()
        attn_close(got, ref.cpu().double().numpy())
        attn_close(got, oracle_attention(cache, q, lens_list, sb))


def test_noalloc_refuses_batches_beyond_its_scratch(kvlib):
    kv = kvlib
    cfg = kv.make_config(32, 8, 32, 3, synth.sign_bits(1))
    batch = 8192                      # needs far more than the 16 MiB scratch
    q = torch.zeros(1, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(q.data_ptr())
    r = kv.lib().kvarn_decode_attn_noalloc(ctypes.byref(cfg), p, 1, p, 1, p, p, 4, p, batch, p, None,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert r == kv._abi.ERR_WORKSPACE
