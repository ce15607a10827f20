"""The 3- and 4-bit code widths on the GPU against the fp64 oracle: bulk
quantise (staged hand-off), dequantise, quantise-on-append, the error split
and split-K decode attention over a ragged paged cache, each over the GPU's
own bytes."""
import zlib
from collections import Counter

import numpy as np
import pytest
import torch

import oracle
import synth
from kvtest_util import PagedCache, assert_code_flip_rate, attn_close, oracle_attention, staged_quantize_parity

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(params=[3, 4], ids=["3bit", "4bit"])
def BITS(request):
    return request.param


def _quantize(kv, cfg, kind, x):
    n = x.shape[0]
    dst = torch.zeros(n * kv.head_block_bytes(cfg), dtype=torch.uint8, device="cuda")
    ws = kv.alloc_workspace(cfg, 0, 0)
    kv.quantize_block(cfg, kind, x.cuda().contiguous(), dst, ws)
    torch.cuda.synchronize()
    return dst.view(n, -1).cpu().numpy(), kv.read_error(ws)


@pytest.mark.parametrize("name,B,iters,dtype,n", [
    ("b32-fp32", 32, 3, "fp32", 16),
    ("b32-bf16", 32, 3, "bf16", 128),
    ("b64-bf16", 64, 2, "bf16", 64),
])
def test_quantize_matches_oracle_staged(kvlib, name, B, iters, dtype, n, BITS):
    kv = kvlib
    sb = synth.sign_bits(B + 40)
    cfg = kv.make_config(4, 1, B, iters, sb, bits=BITS)
    g = synth.make_gen(zlib.crc32(name.encode()) & 0xFFFF)
    x = synth.kv_values(g, 1, n, B, 1.5, 4, 20.0)[0]
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    X = x.double().numpy()
    total = Counter()
    for kind in (0, 1):
        got, err = _quantize(kv, cfg, kind, x)
        assert err == 0
        st = staged_quantize_parity(X, got, B, iters, kind, sb, bits=BITS)
        print(name, kind, dict(st))
        total.update(st)
        assert int(oracle.unpack(B, kind, got[0], bits=BITS)["codes"].max()) <= (1 << BITS) - 1
    assert_code_flip_rate(total)


def test_degenerate_blocks_and_token_scaling(kvlib, BITS):
    """An all-zero block stores zero codes and steps and R = 1; a constant
    block passes the staged check; scaling one token by 8 scales its R by
    exactly 8 and leaves every code and C unchanged."""
    kv = kvlib
    B = 32
    sb = synth.sign_bits(7)
    cfg = kv.make_config(4, 1, B, 3, sb, bits=BITS)
    x = torch.stack([torch.zeros(B, D), torch.full((B, D), 0.75)])
    got, err = _quantize(kv, cfg, 0, x)
    assert err == 0
    staged_quantize_parity(x.double().numpy(), got, B, 3, 0, sb, bits=BITS)
    f = oracle.unpack(B, 0, got[0], bits=BITS)
    assert np.all(f["codes"] == 0) and np.all(f["s16"] == 0) and np.all(f["R16"] == 1)
    g = synth.make_gen(12)
    y = synth.kv_values(g, 1, 1, B, 1.5, 4, 20.0)[0].to(torch.bfloat16).float()
    y2 = y.clone()
    y2[0, 9] *= 8.0
    a, _ = _quantize(kv, cfg, 1, y)
    b, _ = _quantize(kv, cfg, 1, y2)
    fa, fb = oracle.unpack(B, 1, a[0], bits=BITS), oracle.unpack(B, 1, b[0], bits=BITS)
    assert fb["R16"][9] == 8 * fa["R16"][9]
    assert np.array_equal(fa["codes"], fb["codes"]) and np.array_equal(fa["C16"], fb["C16"])


@pytest.mark.parametrize("B", [32, 64])
def test_dequantize_matches_oracle_decode(kvlib, B, BITS):
    kv = kvlib
    sb = synth.sign_bits(11 + B)
    cfg = kv.make_config(4, 1, B, 2, sb, bits=BITS)
    g = synth.make_gen(78 + B)
    x = synth.kv_values(g, 1, 12, B, 1.5, 4, 20.0)[0].to(torch.bfloat16)
    for kind in (0, 1):
        got, _ = _quantize(kv, cfg, kind, x)
        src = torch.from_numpy(got.reshape(-1)).cuda()
        for rotated in (True, False):
            out = torch.empty(12, B, D, dtype=torch.float32, device="cuda")
            kv.dequantize(cfg, kind, src, out, rotated)
            ref = oracle.decode_blocks(got, B, kind, sb, rotated, bits=BITS)
            o = out.cpu().double().numpy()
            scale = np.abs(ref).max(axis=2, keepdims=True) + 1e-30
            assert np.max(np.abs(o - ref) / scale) < 2e-6


def test_wider_codes_reconstruct_better(kvlib):
    """On the same rows every extra bit cuts the reconstruction error (each
    step count is 2^bits - 1: 3, 7, 15)."""
    kv = kvlib
    B = 32
    sb = synth.sign_bits(5)
    g = synth.make_gen(99)
    x = synth.kv_values(g, 1, 32, B, 1.5, 4, 20.0)[0]
    errs = {}
    for bits in (2, 3, 4):
        cfg = kv.make_config(4, 1, B, 3, sb, bits=bits)
        got, _ = _quantize(kv, cfg, 0, x)
        out = torch.empty(32, B, D, dtype=torch.float32, device="cuda")
        kv.dequantize(cfg, 0, torch.from_numpy(got.reshape(-1)).cuda(), out, False)
        xr = out.cpu().double().numpy()
        errs[bits] = np.linalg.norm(xr - x.double().numpy()) / np.linalg.norm(x.double().numpy())
    assert errs[4] < 0.6 * errs[3] and errs[3] < 0.6 * errs[2], errs


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2)])
def test_append_token_by_token(kvlib, B, iters, BITS):
    kv = kvlib
    n_q, n_kv, batch = 4, 2, 2
    sb = synth.sign_bits(B + 3)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb, bits=BITS)
    steps = 2 * B + 3
    g = synth.make_gen(B + 5)
    K = synth.kv_values(g, batch, n_kv, steps, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, steps, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, 3, perm_seed=B)
    ws = kv.alloc_workspace(cfg, 0, 0)
    for s in range(steps):
        pos = torch.full((batch,), s, dtype=torch.int32, device="cuda")
        kn = K[:, :, s].contiguous()
        vn = V[:, :, s].contiguous()
        kv.append(cfg, cache.pool, cache.staging, cache.block_table, pos, kn, vn, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    hb = kv.head_block_bytes(cfg)
    total = Counter()
    for b in range(batch):
        tail = steps % B
        for kind, T in ((0, K), (1, V)):
            assert torch.equal(cache.staging[b, :, kind, :tail], T[b, :, steps - tail:steps])
        for j in range(steps // B):
            for h in range(n_kv):
                for kind, T in ((0, K), (1, V)):
                    rows = T[b, h, j * B:(j + 1) * B].contiguous()
                    dst = torch.zeros(hb, dtype=torch.uint8, device="cuda")
                    kv.quantize_block(cfg, kind, rows[None], dst, ws)
                    torch.cuda.synchronize()
                    got = cache.head_block(b, h, j, kind)
                    assert np.array_equal(got, dst.cpu().numpy())
                    total.update(staged_quantize_parity(rows.double().cpu().numpy()[None], got[None], B,
                                                        iters, kind, sb, bits=BITS))
    assert_code_flip_rate(total)


@pytest.mark.parametrize("B", [32, 64])
def test_error_split_matches_oracle(kvlib, B, BITS):
    kv = kvlib
    sb = synth.sign_bits(610 + B)
    cfg = kv.make_config(4, 1, B, 2, sb, bits=BITS)
    g = synth.make_gen(611 + B, "cuda")
    n = 8
    X = synth.kv_values(g, 1, n, B, 1.5, 4, 20.0, "cuda")[0].contiguous()
    X[2] = 0
    ws = kv.alloc_workspace(cfg, 0, 0)
    Xd = X.double().cpu().numpy()
    for kind in (0, 1):
        pk = torch.zeros(n * kv.head_block_bytes(cfg), dtype=torch.uint8, device="cuda")
        kv.quantize_block(cfg, kind, X, pk, ws)
        out = torch.empty(n, B, 4, device="cuda")
        kv.error_decomposition(cfg, kind, X, pk, out)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        ref = oracle.error_decomposition(Xd, pk.view(n, -1).cpu().numpy(), B, kind, sb, bits=BITS)
        scale = np.maximum(ref[..., 0:1], ref[..., 1:2]) + 1e-30
        np.testing.assert_allclose(got[..., :2], ref[..., :2], rtol=2e-6, atol=1e-30)
        assert np.all(np.abs(got[..., 2:] - ref[..., 2:]) <= 2e-5 * scale + 1e-4 * ref[..., 2:])
        assert np.all(got[2] == 0.0)


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2)])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float32])
def test_attention_ragged_paged_with_tails(kvlib, B, iters, qdtype, BITS):
    kv = kvlib
    n_q, n_kv = 8, 2
    lens = [0, 1, B - 1, B, B + 1, 3 * B + 7, 700]
    batch = len(lens)
    max_blocks = (max(lens) + B - 1) // B + 1
    sb = synth.sign_bits(200 + B)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb, bits=BITS)
    g = synth.make_gen(B + 17)
    K = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(qdtype).cuda()
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=B + 1)
    cache.prefill(K, V, lens)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.full((batch, n_q, D), float("nan"), device="cuda")
    ws = kv.alloc_workspace(cfg, batch, max_blocks)
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    got = out.cpu().double().numpy()
    ref = oracle_attention(cache, q, lens, sb)
    assert np.all(got[0] == 0.0)
    attn_close(got, ref)


@pytest.mark.parametrize("G", [1, 3, 4])
def test_attention_group_sizes_and_long_context(kvlib, G, BITS):
    """Several query heads per kv head, 2048 tokens, B = 64: many blocks per
    warp, so the split-K partials and the merge both run."""
    kv = kvlib
    B, n_kv, batch, L = 64, 2, 3, 2048
    n_q = G * n_kv
    sb = synth.sign_bits(300 + G)
    cfg = kv.make_config(n_q, n_kv, B, 2, sb, bits=BITS)
    g = synth.make_gen(301 + G)
    K = synth.kv_values(g, batch, n_kv, L, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, L, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(torch.bfloat16).cuda()
    lens = [L, L - 5, 97]
    cache = PagedCache(kv, cfg, batch, L // B, perm_seed=G)
    cache.prefill(K, V, lens)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.empty(batch, n_q, D, device="cuda")
    ws = kv.alloc_workspace(cfg, batch, L // B)
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    attn_close(out.cpu().double().numpy(), oracle_attention(cache, q, lens, sb))
