"""GPU decode attention over the 2-bit paged cache (and the bf16 comparison
kernel) against the fp64 oracle over the same cache bytes."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from kvtest_util import PagedCache, attn_close, bf16_bits, oracle_attention

pytestmark = pytest.mark.gpu
D = 128


def _run_attn(kv, cache, q, seq_lens):
    cfg = cache.cfg
    sl = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    out = torch.full((q.shape[0], cfg.n_q_heads, D), float("nan"), device="cuda")
    ws = kv.alloc_workspace(cfg, q.shape[0], cache.max_blocks)
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), kv.read_error(ws)


def test_tiny_single_head(kvlib):
    """One kv head, 256 fp32 tokens (8 blocks of 32), 3 iterations, fp32 query."""
    kv = kvlib
    w = synth.TINY
    sb = synth.sign_bits(w.seed)
    cfg = kv.make_config(w.n_q, w.n_kv, w.block, w.iters, sb)
    g = synth.make_gen(w.seed)
    K = synth.kv_values(g, 1, 1, w.ctx, w.sigma_m, w.n_out, w.out_factor).cuda()
    V = synth.kv_values(g, 1, 1, w.ctx, w.sigma_m, w.n_out, w.out_factor).cuda()
    q = synth.queries(g, 1, 1).cuda()
    cache = PagedCache(kv, cfg, 1, w.ctx // w.block)
    cache.prefill(K, V, [w.ctx])
    got, err = _run_attn(kv, cache, q, [w.ctx])
    assert err == 0
    ref = oracle_attention(cache, q, [w.ctx], sb)
    attn_close(got, ref)


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2)])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float32])
def test_ragged_paged_with_tails(kvlib, B, iters, qdtype):
    kv = kvlib
    n_q, n_kv = 8, 2
    lens = [0, 1, B - 1, B, B + 1, 3 * B + 7, 700]
    batch = len(lens)
    max_blocks = (max(lens) + B - 1) // B + 1
    sb = synth.sign_bits(100 + B)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb)
    g = synth.make_gen(B)
    K = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(qdtype).cuda()
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=B)
    cache.prefill(K, V, lens)
    got, err = _run_attn(kv, cache, q, lens)
    assert err == 0
    ref = oracle_attention(cache, q, lens, sb)
    assert np.all(got[0] == 0.0)            # empty sequence -> zeros
    attn_close(got, ref)


@pytest.mark.parametrize("batch", [24, 16])
@pytest.mark.parametrize("B", [32, 64])
def test_merge_paths_with_tails(kvlib, B, batch):
    """32 query heads over 8 kv heads, every sequence with raw tail rows (1 to
    3 blocks and a tail of 1 .. B - 1 rows). 24 sequences: more rows than one
    wave of the wide merge holds (4 CTAs per SM) and fewer split warps than
    16 per unit, so the one-warp-per-row merge scores the tails. 16
    sequences: 512 rows fit one wave, so the 8-warp merge takes them, its
    warps loading 4 partials per round trip. Sampled sequences against the
    oracle."""
    kv = kvlib
    n_q, n_kv = 32, 8
    lens = [B * (1 + i % 3) + 1 + (7 * i) % (B - 1) for i in range(batch)]
    assert all(L % B for L in lens)
    max_blocks = max(lens) // B + 1
    sb = synth.sign_bits(300 + B)
    cfg = kv.make_config(n_q, n_kv, B, 2, sb)
    g = synth.make_gen(300 + B + batch)
    K = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=B + 1)
    cache.prefill(K, V, lens)
    got, err = _run_attn(kv, cache, q, lens)
    assert err == 0
    seqs = [0, 7, batch - 1]
    ref = oracle_attention(cache, q, lens, sb, seqs=seqs)
    attn_close(got[seqs], ref)


@pytest.mark.parametrize("G", [1, 2, 3, 4])
@pytest.mark.parametrize("B", [32, 64])
def test_group_sizes(kvlib, G, B):
    """G = n_q / n_kv query heads per kv head (empty columns and, at B = 64,
    empty rows of the shared-memory q planes for G < 4)."""
    kv = kvlib
    n_kv = 2
    n_q = G * n_kv
    lens = [5 * B + 3, 2 * B]
    sb = synth.sign_bits(G)
    cfg = kv.make_config(n_q, n_kv, B, 3, sb)
    g = synth.make_gen(40 + G)
    K = synth.kv_values(g, 2, n_kv, max(lens), 1.0, 2, 10.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, 2, n_kv, max(lens), 1.0, 2, 10.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, 2, n_q).cuda()
    cache = PagedCache(kv, cfg, 2, 8, perm_seed=G)
    cache.prefill(K, V, lens)
    got, err = _run_attn(kv, cache, q, lens)
    assert err == 0
    attn_close(got, oracle_attention(cache, q, lens, sb))


def test_closed_form_uniform_keys(kvlib):
    """All keys equal (constant block) -> uniform weights -> mean of the values."""
    kv = kvlib
    B, n_kv, n_q = 32, 1, 4
    sb = synth.sign_bits(8)
    cfg = kv.make_config(n_q, n_kv, B, 3, sb)
    L = 4 * B
    K = torch.ones(1, 1, L, D).cuda() * 0.5
    g = synth.make_gen(8)
    V = synth.kv_values(g, 1, 1, L, 1.0, 2, 10.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, 1, n_q).cuda()
    cache = PagedCache(kv, cfg, 1, 4)
    cache.prefill(K, V, [L])
    got, _ = _run_attn(kv, cache, q, [L])
    vhat = np.concatenate([oracle.decode_blocks(cache.head_block(0, 0, j, 1), B, 1, sb, False)[0]
                           for j in range(4)])
    for j in range(n_q):
        attn_close(got[0, j], vhat.mean(axis=0))


def test_bad_block_id_and_length_are_flagged(kvlib):
    kv = kvlib
    B = 32
    sb = synth.sign_bits(2)
    cfg = kv.make_config(4, 1, B, 3, sb)
    g = synth.make_gen(2)
    K = synth.kv_values(g, 2, 1, 3 * B, 1.0, 2, 10.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, 2, 3)
    cache.prefill(K, K, [3 * B, 3 * B])
    q = synth.queries(g, 2, 4).cuda()
    cache.block_table[0, 1] = 10_000          # outside the pool
    _, err = _run_attn(kv, cache, q, [3 * B, 3 * B])
    assert err & kv.DEVERR_BLOCK_ID
    cache.block_table[0, 1] = 1
    got, err = _run_attn(kv, cache, q, [3 * B, 10 * B])   # beyond the table
    assert err & kv.DEVERR_POSITION
    assert np.all(np.isnan(got[1]))


def test_bf16_cache_kernel(kvlib):
    """The comparison kernel: same attention over a plain bf16 paged cache."""
    kv = kvlib
    for B in (32, 64):
        n_q, n_kv = 8, 2
        lens = [1, 17, B, 5 * B + 9, 300]
        batch = len(lens)
        max_blocks = (max(lens) + B - 1) // B
        cfg = kv.make_config(n_q, n_kv, B, 3, synth.sign_bits(0))
        g = synth.make_gen(60 + B)
        K = synth.kv_values(g, batch, n_kv, max_blocks * B, 1.5, 4, 20.0).to(torch.bfloat16)
        V = synth.kv_values(g, batch, n_kv, max_blocks * B, 1.5, 4, 20.0).to(torch.bfloat16)
        q = synth.queries(g, batch, n_q).cuda()
        perm = np.random.default_rng(B).permutation(batch * max_blocks).astype(np.int32)
        bt = perm.reshape(batch, max_blocks)
        # rows past each sequence's length hold NaN: the kernel must never let them in
        pool = torch.full((batch * max_blocks, n_kv, 2, B, D), float("nan"), dtype=torch.bfloat16)
        for b in range(batch):
            for j in range(max_blocks):
                n = min(B, max(0, lens[b] - j * B))
                pool[bt[b, j], :, 0, :n] = K[b, :, j * B:j * B + n]
                pool[bt[b, j], :, 1, :n] = V[b, :, j * B:j * B + n]
        out = torch.empty(batch, n_q, D, device="cuda")
        ws = kv.alloc_workspace(cfg, batch, max_blocks)
        kv.decode_attn_bf16(cfg, q, pool.cuda(), torch.from_numpy(bt).cuda(),
                            torch.tensor(lens, dtype=torch.int32, device="cuda"), out, ws)
        torch.cuda.synchronize()
        assert kv.read_error(ws) == 0
        got = out.cpu().double().numpy()
        Kd, Vd, qd = K.double().numpy(), V.double().numpy(), q.double().cpu().numpy()
        G = n_q // n_kv
        for b in range(batch):
            for j in range(n_q):
                ref = oracle.attention(qd[b, j], Kd[b, j // G, :lens[b]], Vd[b, j // G, :lens[b]],
                                       1 / math.sqrt(D))
                attn_close(got[b, j], ref)


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2)])
def test_small_call_after_large_on_one_workspace(kvlib, B, iters):
    """A workload with fewer blocks than resident warps, run on a workspace a
    large call has just filled with partials: the merge must read only the
    partials of warps that own blocks of each unit (stale slots of the
    earlier call must not leak in), for the 2-bit and the bf16 kernel."""
    kv = kvlib
    n_q, n_kv = 32, 8
    sb = synth.sign_bits(7 + B)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb)
    g = synth.make_gen(900 + B)
    big_batch, big_len = 16, 64 * B       # 16 * 8 * 64 blocks: more than the resident warps
    small_lens = [3 * B + 5]
    ws = kv.alloc_workspace(cfg, big_batch, 64)
    # ---- large call: fills every partial slot with its own data
    Kb = synth.kv_values(g, big_batch, n_kv, big_len, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    Vb = synth.kv_values(g, big_batch, n_kv, big_len, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    big = PagedCache(kv, cfg, big_batch, 64, perm_seed=1)
    big.prefill(Kb, Vb, [big_len] * big_batch)
    del Kb, Vb
    qb = synth.queries(g, big_batch, n_q).to(torch.bfloat16).cuda()
    out_b = torch.empty(big_batch, n_q, D, device="cuda")
    kv.decode_attn(cfg, qb, big.pool, big.staging, big.block_table,
                   torch.full((big_batch,), big_len, dtype=torch.int32, device="cuda"), out_b, ws)
    # ---- small call on the same workspace
    Ks = synth.kv_values(g, 1, n_kv, small_lens[0], 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    Vs = synth.kv_values(g, 1, n_kv, small_lens[0], 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    small = PagedCache(kv, cfg, 1, 4, perm_seed=2)
    small.prefill(Ks, Vs, small_lens)
    qs = synth.queries(g, 1, n_q).to(torch.bfloat16).cuda()
    out_s = torch.full((1, n_q, D), float("nan"), device="cuda")
    kv.decode_attn(cfg, qs, small.pool, small.staging, small.block_table,
                   torch.tensor(small_lens, dtype=torch.int32, device="cuda"), out_s, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    attn_close(out_s.cpu().double().numpy(), oracle_attention(small, qs, small_lens, sb))
    # ---- the bf16 kernel on the same workspace, after another large call
    kvp_big = torch.randn(big_batch * 64, n_kv, 2, B, D, device="cuda").to(torch.bfloat16)
    btb = torch.arange(big_batch * 64, dtype=torch.int32, device="cuda").view(big_batch, 64)
    kv.decode_attn_bf16(cfg, qb, kvp_big, btb,
                        torch.full((big_batch,), big_len, dtype=torch.int32, device="cuda"), out_b, ws)
    L = small_lens[0]
    nb = (L + B - 1) // B
    kvp = torch.zeros(nb, n_kv, 2, B, D, dtype=torch.bfloat16)
    for j in range(nb):
        n = min(B, L - j * B)
        kvp[j, :, 0, :n] = Ks[0, :, j * B:j * B + n].cpu()
        kvp[j, :, 1, :n] = Vs[0, :, j * B:j * B + n].cpu()
    kv.decode_attn_bf16(cfg, qs, kvp.cuda(), torch.arange(nb, dtype=torch.int32, device="cuda").view(1, nb),
                        torch.tensor(small_lens, dtype=torch.int32, device="cuda"), out_s, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    got = out_s.cpu().double().numpy()
    Kd, Vd, qd = Ks.double().cpu().numpy(), Vs.double().cpu().numpy(), qs.double().cpu().numpy()
    for j in range(n_q):
        ref = oracle.attention(qd[0, j], Kd[0, j // 4, :L], Vd[0, j // 4, :L], 1 / math.sqrt(D))
        attn_close(got[0, j], ref)


@pytest.mark.parametrize("B", [32, 64])
def test_wait_timeout_path_flags_and_workspace_stays_usable(kvlib, B):
    """The bounded copy wait run out on purpose (the test switch gives every
    warp's first wait a limit of zero): the call raises
    KVARN_DEVERR_WAIT_TIMEOUT and returns without hanging, the copies in
    flight are waited for, and after the error word is cleared the next call
    on the same workspace matches the oracle."""
    kv = kvlib
    n_q, n_kv = 8, 2
    lens = [5 * B + 3, 9 * B, 2 * B + B // 2, 1]
    batch = len(lens)
    sb = synth.sign_bits(77 + B)
    cfg = kv.make_config(n_q, n_kv, B, 3, sb)
    cfg_t = kv.make_config(n_q, n_kv, B, 3, sb, flags=kv.FLAG_TEST_WAIT_TIMEOUT)
    g = synth.make_gen(77)
    K = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, (max(lens) + B - 1) // B, perm_seed=7)
    cache.prefill(K, V, lens)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = kv.alloc_workspace(cfg, batch, cache.max_blocks)
    out = torch.zeros(batch, n_q, D, device="cuda")
    for _ in range(2):
        kv.decode_attn(cfg_t, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
        assert kv.read_error(ws) & kv.DEVERR_WAIT_TIMEOUT
        kv.clear_error(ws)
    out = torch.full((batch, n_q, D), float("nan"), device="cuda")
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    assert kv.read_error(ws) == 0
    attn_close(out.cpu().double().numpy(), oracle_attention(cache, q, lens, sb))
