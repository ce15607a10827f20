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


def test_bench_step_state_after_replays_matches_the_oracle(kvlib):
    """The benchmark's own step on the Qwen3-4B workload (two of its layers at
    full size, built by bench.py's recipe), captured as a CUDA graph and
    replayed: afterwards the block every append completed and the attention
    output of sampled sequences of the last layer match the oracle over the
    GPU's cache bytes."""
    import bench
    import oracle
    from kvtest_util import assert_code_flip_rate, attn_close, bf16_bits, staged_quantize_parity
    from collections import Counter
    kv = kvlib
    w = synth.QWEN3_4B_CACHE
    state = bench.build_layers(kv, w, 2, "cuda")
    B, nb = w.block, w.ctx // w.block
    ws = kv.alloc_workspace(state[0]["cfg"], w.batch, nb)
    pos = torch.full((w.batch,), w.ctx - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((w.batch,), w.ctx, dtype=torch.int32, device="cuda")
    out = torch.full((2, w.batch, w.n_q, D), float("nan"), device="cuda")

    def step():
        for l, st in enumerate(state):
            kv.append(st["cfg"], st["pool"], st["staging"], st["bt"], pos, st["k_new"], st["v_new"], ws)
            kv.decode_attn(st["cfg"], st["q"], st["pool"], st["staging"], st["bt"], lens, out[l], ws)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert kv.read_error(ws) == 0
    st = state[1]
    sb = [int(x) for x in st["cfg"].sign_bits]
    pool_np = st["pool"].cpu().numpy()
    bt_np = st["bt"].cpu().numpy()
    hb, bb = kv.head_block_bytes(st["cfg"]), kv.block_bytes(st["cfg"])
    # the completed block of (sequence 63, kv head 5): staged rows + the appended one
    b, h = 63, 5
    total = Counter()
    for kind, new in ((0, st["k_new"]), (1, st["v_new"])):
        rows = np.concatenate([oracle.bf16_array_to_f64(bf16_bits(st["staging"][b, h, kind, :B - 1])),
                               oracle.bf16_array_to_f64(bf16_bits(new[b, h][None]))])
        o = int(bt_np[b, nb - 1]) * bb + (2 * h + kind) * hb
        total.update(staged_quantize_parity(rows[None], pool_np.reshape(-1)[o:o + hb][None], B, w.iters, kind, sb))
    assert_code_flip_rate(total)
    seqs = [0, 37, 63]
    qn = st["q"][seqs].double().cpu().numpy()
    ref = oracle.decode_attention(B, w.n_q, w.n_kv, sb, 1.0 / np.sqrt(D), qn, pool_np,
                                  bf16_bits(st["staging"][seqs]), np.ascontiguousarray(bt_np[seqs]),
                                  np.full(len(seqs), w.ctx, dtype=np.int32))
    attn_close(out[1].cpu().double().numpy()[seqs], ref)
