"""GPU quantise-on-append: staging rows, block completion into the paged pool
(identical bytes to the bulk quantiser on the same rows, oracle parity)."""
import numpy as np
import pytest
import torch

import synth
from collections import Counter

from kvtest_util import PagedCache, assert_code_flip_rate, staged_quantize_parity

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2)])
def test_append_token_by_token(kvlib, B, iters):
    kv = kvlib
    n_q, n_kv, batch = 4, 2, 3
    sb = synth.sign_bits(B)
    cfg = kv.make_config(n_q, n_kv, B, iters, sb)
    steps = 2 * B + 5
    g = synth.make_gen(B + 1)
    K = synth.kv_values(g, batch, n_kv, steps, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    V = synth.kv_values(g, batch, n_kv, steps, 1.5, 4, 20.0).to(torch.bfloat16).cuda()
    cache = PagedCache(kv, cfg, batch, 4, perm_seed=B)
    ws = kv.alloc_workspace(cfg, 0, 0)
    start = [0, 3, B - 1]        # sequences at different positions
    for s in range(steps - max(start)):
        pos = torch.tensor([p + s for p in start], dtype=torch.int32, device="cuda")
        kn = torch.stack([K[b, :, start[b] + s] for b in range(batch)]).contiguous()
        vn = torch.stack([V[b, :, start[b] + s] for b in range(batch)]).contiguous()
        kv.append(cfg, cache.pool, cache.staging, cache.block_table, pos, kn, vn, ws)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    hb = kv.head_block_bytes(cfg)
    total = Counter()
    for b in range(batch):
        L = start[b] + steps - max(start)
        # staging holds the rows of the open block (raw)
        tail = L % B
        for kind, T in ((0, K), (1, V)):
            assert torch.equal(cache.staging[b, :, kind, :tail], T[b, :, L - tail:L])
        for j in range(L // B):
            if (j + 1) * B <= start[b]:
                continue                      # block never appended here
            for h in range(n_kv):
                for kind, T in ((0, K), (1, V)):
                    rows = T[b, h, j * B:(j + 1) * B].contiguous()
                    dst = torch.zeros(hb, dtype=torch.uint8, device="cuda")
                    kv.quantize_block(cfg, kind, rows[None], dst, ws)
                    torch.cuda.synchronize()
                    got = cache.head_block(b, h, j, kind)
                    if (j * B) >= start[b]:
                        assert np.array_equal(got, dst.cpu().numpy())
                        total.update(staged_quantize_parity(rows.double().cpu().numpy()[None], got[None], B,
                                                            iters, kind, sb))
    assert_code_flip_rate(total)


def test_append_position_out_of_range(kvlib):
    kv = kvlib
    cfg = kv.make_config(4, 1, 32, 3, synth.sign_bits(1))
    cache = PagedCache(kv, cfg, 1, 2)
    ws = kv.alloc_workspace(cfg, 0, 0)
    kn = torch.zeros(1, 1, D, dtype=torch.bfloat16, device="cuda")
    kv.append(cfg, cache.pool, cache.staging, cache.block_table,
              torch.tensor([64], dtype=torch.int32, device="cuda"), kn, kn, ws)
    assert kv.read_error(ws) & kv.DEVERR_POSITION
    kv.clear_error(ws)
    cache.block_table[0, 0] = -5
    kv.append(cfg, cache.pool, cache.staging, cache.block_table,
              torch.tensor([31], dtype=torch.int32, device="cuda"), kn, kn, ws)
    assert kv.read_error(ws) & kv.DEVERR_BLOCK_ID
