"""GPU quantise / dequantise parity with the fp64 oracle (staged hand-off)."""
import zlib
from collections import Counter

import numpy as np
import pytest
import torch

import oracle
import synth
from kvtest_util import assert_code_flip_rate, staged_quantize_parity

pytestmark = pytest.mark.gpu
D = 128


def _values(seed, n, B, sigma_m, n_out, factor, dtype):
    g = synth.make_gen(seed)
    x = synth.kv_values(g, 1, n, B, sigma_m, n_out, factor)[0]          # [n][B][128]
    return x.to(torch.bfloat16) if dtype == "bf16" else x


def _quantize(kv, cfg, kind, x):
    n = x.shape[0]
    dst = torch.zeros(n * kv.head_block_bytes(cfg), dtype=torch.uint8, device="cuda")
    ws = kv.alloc_workspace(cfg, 0, 0)
    kv.quantize_block(cfg, kind, x.cuda().contiguous(), dst, ws)
    torch.cuda.synchronize()
    return dst.view(n, -1).cpu().numpy(), kv.read_error(ws)


@pytest.mark.parametrize("name,B,iters,dtype,n,sigma_m,n_out,factor", [
    ("tiny-fp32", 32, 3, "fp32", 8, 1.0, 2, 10.0),
    ("llama-bf16", 32, 3, "bf16", 96, 1.5, 4, 20.0),
    ("qwen-bf16", 64, 2, "bf16", 48, 1.5, 4, 20.0),
    ("iters1", 32, 1, "bf16", 16, 1.5, 4, 20.0),
    ("llama-bf16-2M-codes", 32, 3, "bf16", 256, 1.5, 4, 20.0),
    ("iters4-b64", 64, 4, "bf16", 16, 1.0, 2, 10.0),
])
def test_quantize_matches_oracle_staged(kvlib, name, B, iters, dtype, n, sigma_m, n_out, factor):
    kv = kvlib
    sb = synth.sign_bits(B + iters)
    cfg = kv.make_config(4, 1, B, iters, sb)
    x = _values(zlib.crc32(name.encode()) & 0xFFFF, n, B, sigma_m, n_out, factor, dtype)
    X = x.double().numpy()
    total = Counter()
    for kind in (0, 1):
        got, err = _quantize(kv, cfg, kind, x)
        assert err == 0
        st = staged_quantize_parity(X, got, B, iters, kind, sb)
        print(name, kind, dict(st))
        total.update(st)
    assert_code_flip_rate(total)


def test_dequantize_matches_oracle_decode(kvlib):
    kv = kvlib
    B, iters = 32, 3
    sb = synth.sign_bits(9)
    cfg = kv.make_config(4, 1, B, iters, sb)
    x = _values(77, 12, B, 1.5, 4, 20.0, "bf16")
    for kind in (0, 1):
        got, _ = _quantize(kv, cfg, kind, x)
        src = torch.from_numpy(got.reshape(-1)).cuda()
        for rotated in (True, False):
            out = torch.empty(12, B, D, dtype=torch.float32, device="cuda")
            kv.dequantize(cfg, kind, src, out, rotated)
            ref = oracle.decode_blocks(got, B, kind, sb, rotated)
            o = out.cpu().double().numpy()
            scale = np.abs(ref).max(axis=2, keepdims=True) + 1e-30
            assert np.max(np.abs(o - ref) / scale) < 2e-6


def test_offsets_and_strides(kvlib):
    """Interleaved source rows (token stride 256) and scattered destinations."""
    kv = kvlib
    B, iters = 32, 3
    sb = synth.sign_bits(3)
    cfg = kv.make_config(4, 1, B, iters, sb)
    n = 10
    x = _values(5, 2 * n, B, 1.5, 4, 20.0, "bf16").view(n, 2, B, D).transpose(1, 2).contiguous()  # [n][B][2][128]
    hb = kv.head_block_bytes(cfg)
    perm = np.random.default_rng(0).permutation(n)
    offs = torch.tensor(perm * hb, dtype=torch.int64, device="cuda")
    dst = torch.zeros(n * hb, dtype=torch.uint8, device="cuda")
    ws = kv.alloc_workspace(cfg, 0, 0)
    xs = x.cuda()
    kv.quantize_block(cfg, 1, xs[:, :, 1], dst, ws, dst_offsets=offs, n_head_blocks=n,
                      block_stride=B * 2 * D, token_stride=2 * D)
    torch.cuda.synchronize()
    want, _ = _quantize(kv, cfg, 1, x[:, :, 1].contiguous())
    got = dst.view(n, hb).cpu().numpy()
    for i in range(n):
        assert np.array_equal(got[perm[i]], want[i])


def test_degenerate_blocks_and_nonfinite_flag(kvlib):
    kv = kvlib
    B = 32
    sb = synth.sign_bits(4)
    cfg = kv.make_config(4, 1, B, 3, sb)
    zeros = torch.zeros(1, B, D)
    const = torch.full((1, B, D), 0.75)
    got, err = _quantize(kv, cfg, 0, torch.cat([zeros, const]))
    assert err == 0
    X = torch.cat([zeros, const]).double().numpy()
    staged_quantize_parity(X, got, B, 3, 0, sb)
    f = oracle.unpack(B, 0, got[0])
    assert np.all(f["codes"] == 0) and np.all(f["s16"] == 0) and np.all(f["R16"] == 1)
    bad = torch.randn(1, B, D)
    bad[0, 3, 7] = float("nan")
    _, err = _quantize(kv, cfg, 0, bad)
    assert err & kv.DEVERR_NONFINITE


def test_token_scaling_is_exact_on_gpu(kvlib):
    kv = kvlib
    B = 32
    sb = synth.sign_bits(6)
    cfg = kv.make_config(4, 1, B, 3, sb)
    x = _values(12, 1, B, 1.5, 4, 20.0, "bf16").float()
    x2 = x.clone()
    x2[0, 9] *= 8.0
    a, _ = _quantize(kv, cfg, 0, x)
    b, _ = _quantize(kv, cfg, 0, x2)
    fa, fb = oracle.unpack(B, 0, a[0]), oracle.unpack(B, 0, b[0])
    assert fb["R16"][9] == 8 * fa["R16"][9]
    assert np.array_equal(fa["codes"], fb["codes"]) and np.array_equal(fa["C16"], fb["C16"])
