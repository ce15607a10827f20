"""A multi-layer decode step (append + attention per layer) captured once as
a CUDA graph and replayed gives the same cache bytes and outputs as the same
calls issued one by one: the entry points only enqueue kernels on the
caller's stream, so a serving loop can capture them."""
import numpy as np
import pytest
import torch

import synth
from kvtest_util import PagedCache

pytestmark = pytest.mark.gpu
D = 128


def _layers(kv, n_layers, batch, ctx, B):
    out = []
    for l in range(n_layers):
        sb = synth.sign_bits(500 + l)
        cfg = kv.make_config(32, 8, B, 2, sb)
        g = synth.make_gen(500 + l, "cuda")
        K = synth.kv_values(g, batch, 8, ctx, 1.5, 4, 20.0, "cuda").to(torch.bfloat16)
        V = synth.kv_values(g, batch, 8, ctx, 1.5, 4, 20.0, "cuda").to(torch.bfloat16)
        cache = PagedCache(kv, cfg, batch, ctx // B, perm_seed=l)
        cache.prefill(K, V, [ctx - 1] * batch)
        q = synth.queries(g, batch, 32, "cuda").to(torch.bfloat16)
        out.append(dict(cfg=cfg, cache=cache, q=q, k=K[:, :, ctx - 1].contiguous(), v=V[:, :, ctx - 1].contiguous()))
    return out


@pytest.mark.parametrize("B", [32, 64])
def test_captured_decode_step_equals_eager(kvlib, B):
    kv = kvlib
    batch, ctx, n_layers = 4, 8 * B, 4
    layers = _layers(kv, n_layers, batch, ctx, B)
    pos = torch.full((batch,), ctx - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((batch,), ctx, dtype=torch.int32, device="cuda")
    ws = kv.alloc_workspace(layers[0]["cfg"], batch, ctx // B)
    outs = torch.zeros(n_layers, batch, 32, D, device="cuda")

    def step():
        for l, st in enumerate(layers):
            c = st["cache"]
            kv.append(st["cfg"], c.pool, c.staging, c.block_table, pos, st["k"], st["v"], ws)
            kv.decode_attn(st["cfg"], st["q"], c.pool, c.staging, c.block_table, lens, outs[l], ws)

    step()                                  # eager (also fills the launch-size caches)
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    eager = outs.clone()
    pools = [st["cache"].pool.clone() for st in layers]
    outs.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    assert torch.equal(outs, eager)
    for st, p in zip(layers, pools):
        assert torch.equal(st["cache"].pool, p)
    assert np.isfinite(eager.cpu().numpy()).all()
