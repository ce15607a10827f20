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
