"""The per-token magnitude / direction split of the quantisation error on the
GPU against the oracle over the GPU's own packed bytes (K and V layouts,
bf16 and fp32 inputs, with and without rotation, a zero block)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("B,iters,flags", [(32, 3, 0), (64, 2, 0), (32, 3, oracle.NO_ROTATION)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_error_split_matches_oracle(kvlib, B, iters, flags, dtype):
    kv = kvlib
    sb = synth.sign_bits(600 + B)
    cfg = kv.make_config(4, 1, B, iters, sb, flags=flags)
    g = synth.make_gen(601 + B + flags, "cuda")
    n = 16
    X = synth.kv_values(g, 1, n, B, 1.5, 4, 20.0, "cuda")[0].to(dtype).contiguous()
    X[3] = 0                                    # an all-zero block: no error at all
    X[5, 7] = 0                                 # one zero token inside a block
    ws = kv.alloc_workspace(cfg, 0, 0)
    Xd = X.double().cpu().numpy()
    for kind in (0, 1):
        pk = torch.zeros(n * kv.head_block_bytes(cfg), dtype=torch.uint8, device="cuda")
        kv.quantize_block(cfg, kind, X, pk, ws)
        out = torch.empty(n, B, 4, device="cuda")
        kv.error_decomposition(cfg, kind, X, pk, out)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        ref = oracle.error_decomposition(Xd, pk.view(n, -1).cpu().numpy(), B, kind, sb, flags=flags)
        scale = np.maximum(ref[..., 0:1], ref[..., 1:2]) + 1e-30
        assert np.all(np.isfinite(got))
        np.testing.assert_allclose(got[..., :2], ref[..., :2], rtol=2e-6, atol=1e-30)
        assert np.all(np.abs(got[..., 2:] - ref[..., 2:]) <= 2e-5 * scale + 1e-4 * ref[..., 2:])
        assert np.all(got[3] == 0.0)


@pytest.mark.parametrize("bits", [2, 4])
def test_error_split_over_a_paged_pool(kvlib, bits):
    """A [batch][n_kv][L][128] source against its head-blocks scattered over a
    pool by offsets: every one of the batch x n_kv x L/B blocks is written (the
    output starts as NaN) and equals the oracle."""
    kv = kvlib
    B, batch, n_kv, nb = 32, 2, 2, 4
    sb = synth.sign_bits(620 + bits)
    cfg = kv.make_config(4, n_kv, B, 3, sb, bits=bits)
    g = synth.make_gen(621 + bits, "cuda")
    T = synth.kv_values(g, batch, n_kv, nb * B, 1.5, 4, 20.0, "cuda").to(torch.bfloat16).contiguous()
    hb = kv.head_block_bytes(cfg)
    n = batch * n_kv * nb
    perm = torch.from_numpy(np.random.default_rng(bits).permutation(n)).cuda()
    offs = (perm.long() * hb).contiguous()
    pool = torch.zeros(n * hb, dtype=torch.uint8, device="cuda")
    ws = kv.alloc_workspace(cfg, 0, 0)
    kv.quantize_block(cfg, 1, T, pool, ws, dst_offsets=offs, n_head_blocks=n)
    out = torch.full((n, B, 4), float("nan"), device="cuda")
    kv.error_decomposition(cfg, 1, T, pool, out, packed_offsets=offs)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    pk = pool.view(n, hb)[perm.cpu()].cpu().numpy()
    ref = oracle.error_decomposition(T.double().cpu().numpy().reshape(n, B, D), pk, B, 1, sb, bits=bits)
    scale = np.maximum(ref[..., 0:1], ref[..., 1:2]) + 1e-30
    np.testing.assert_allclose(got[..., :2], ref[..., :2], rtol=2e-6, atol=1e-30)
    assert np.all(np.abs(got[..., 2:] - ref[..., 2:]) <= 2e-5 * scale + 1e-4 * ref[..., 2:])
