"""The ablation switches (the pages' 消融 list: Hadamard only, VarN only,
VarN along the token axis only or the channel axis only) on the GPU, each
against the oracle run with the same switches: quantiser bytes (staged
parity), dequantisation, and decode attention over the GPU's own cache."""
import numpy as np
import pytest
import torch

import oracle
import synth
from kvtest_util import PagedCache, assert_code_flip_rate, attn_close, oracle_attention, staged_quantize_parity

pytestmark = pytest.mark.gpu
D = 128

NR, NT, NC = oracle.NO_ROTATION, oracle.NO_TOKEN_PASS, oracle.NO_CHANNEL_PASS
VARIANTS = [  # (name, flags, iters)
    ("hadamard-only", 0, 0),
    ("varn-only", NR, 3),
    ("token-axis-only", NC, 3),
    ("channel-axis-only", NT, 2),
    ("plain-group-2bit", NR, 0),
]


@pytest.mark.parametrize("name,flags,iters", VARIANTS)
@pytest.mark.parametrize("B", [32, 64])
def test_ablation_quantise_and_dequantise(kvlib, name, flags, iters, B):
    kv = kvlib
    assert (kv.FLAG_NO_ROTATION, kv.FLAG_NO_TOKEN_PASS, kv.FLAG_NO_CHANNEL_PASS) == (NR, NT, NC)
    sb = synth.sign_bits(300 + B + flags)
    cfg = kv.make_config(4, 1, B, iters, sb, flags=flags)
    g = synth.make_gen(301 + B + 7 * flags + iters, "cuda")
    n = 24
    X = synth.kv_values(g, 1, n, B, 1.5, 4, 20.0, "cuda")[0].to(torch.bfloat16).contiguous()
    ws = kv.alloc_workspace(cfg, 0, 0)
    Xd = X.double().cpu().numpy()
    from collections import Counter
    tot = Counter()
    for kind in (0, 1):
        dst = torch.zeros(n * kv.head_block_bytes(cfg), dtype=torch.uint8, device="cuda")
        kv.quantize_block(cfg, kind, X, dst, ws)
        torch.cuda.synchronize()
        assert kv.read_error(ws) == 0
        got = dst.view(n, -1).cpu().numpy()
        tot += staged_quantize_parity(Xd, got, B, iters, kind, sb, flags=flags)
        out = torch.empty(n, B, D, device="cuda")
        kv.dequantize(cfg, kind, dst, out, rotated=False)
        ref = oracle.decode_blocks(got, B, kind, sb, rotated=False, flags=flags)
        np.testing.assert_allclose(out.double().cpu().numpy(), ref, rtol=2e-6, atol=2e-6 * np.abs(ref).max())
    assert_code_flip_rate(tot)


@pytest.mark.parametrize("name,flags,iters", VARIANTS)
def test_ablation_decode_attention(kvlib, name, flags, iters):
    kv = kvlib
    B, n_q, n_kv = 32, 8, 2
    lens = [5, B + 3, 4 * B + 17, 300]
    batch = len(lens)
    max_blocks = (max(lens) + B - 1) // B
    sb = synth.sign_bits(400 + flags)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb, flags=flags)
    g = synth.make_gen(401 + flags + iters)
    K = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, max(lens), 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    q = synth.queries(g, batch, n_q).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, max_blocks, perm_seed=flags)
    cache.prefill(K, V, lens)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.empty(batch, n_q, D, device="cuda")
    ws = kv.alloc_workspace(cfg, batch, max_blocks)
    kv.decode_attn(cfg, q, cache.pool, cache.staging, cache.block_table, sl, out, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    attn_close(out.cpu().double().numpy(), oracle_attention(cache, q, lens, sb))
