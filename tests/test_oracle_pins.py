"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: exact
integer identities, closed forms, numpy's own float16 type, brute force over
every fp16 value, hand-derived bytes, or invariants the method states
(rotation keeps norms and cancels in q.k; VarN drives row and column
variances to 1; the kept scales restore the data; the quantiser's error is at
most half a step).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

D = 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pack_patterns.txt")


def _popcount_sign(i, j):
    return -1 if bin(i & j).count("1") % 2 else 1


# ---------------------------------------------------------------- rotation

def test_hadamard_is_sylvester_with_popcount_entries_and_orthogonal():
    H = oracle.hadamard(D).astype(np.int64)
    for n in (1, 2, 4, 8, 16, 32, 64):
        Hn = oracle.hadamard(n).astype(np.int64)
        assert np.array_equal(Hn @ Hn.T, n * np.eye(n, dtype=np.int64))
    assert np.array_equal(H @ H.T, D * np.eye(D, dtype=np.int64))
    ref = np.array([[_popcount_sign(i, j) for j in range(D)] for i in range(D)])
    assert np.array_equal(H, ref)


def test_rotation_of_basis_vectors_matches_closed_form():
    sb = synth.sign_bits(7)
    sig = oracle.sigma(sb)
    E = np.eye(D)
    R_cols = oracle.rotate(E, sb)            # row i = R e_i
    for i in range(D):
        want = np.array([sig[i] * _popcount_sign(j, i) for j in range(D)]) / math.sqrt(D)
        np.testing.assert_allclose(R_cols[i], want, rtol=0, atol=1e-15)


def test_rotation_keeps_norm_and_inverts():
    rng = np.random.default_rng(1)
    sb = synth.sign_bits(3)
    x = rng.standard_normal((20, D)) * np.exp(rng.standard_normal((20, 1)) * 2)
    y = oracle.rotate(x, sb)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    np.testing.assert_allclose(oracle.unrotate(y, sb), x, rtol=0, atol=1e-12 * np.abs(x).max())


def test_signs_apply_before_the_hadamard():
    rng = np.random.default_rng(2)
    sb = synth.sign_bits(11)
    x = rng.standard_normal((4, D))
    zero = np.zeros(4, dtype=np.uint32)
    np.testing.assert_allclose(oracle.rotate(x, sb), oracle.rotate(x * oracle.sigma(sb), zero),
                               atol=1e-14)


def test_sign_bits_are_splitmix64_and_not_degenerate():
    # SplitMix64 from state 0: first output 0xE220A8397B1DCDAF (published test value)
    st, out = synth.splitmix64(0)
    assert out == 0xE220A8397B1DCDAF
    s = oracle.sigma(synth.sign_bits(0))
    assert 40 < (s < 0).sum() < 88


# ---------------------------------------------------------------- fp16 / bf16 grid

def _sample_values(rng, n):
    mag = np.exp(rng.uniform(np.log(1e-9), np.log(7e4), n))
    return mag * rng.choice([-1.0, 1.0], n)


def test_f16_round_nearest_matches_numpy_float16():
    rng = np.random.default_rng(3)
    vals = np.concatenate([_sample_values(rng, 20000),
                           [65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                            1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -0.0, 0.0]])
    for v in vals:
        with np.errstate(over="ignore"):
            want = float(np.float16(v))
        got = oracle.f16_rn(v)
        assert got == want or (math.isinf(got) and math.isinf(want)), (v, got, want)


def test_f16_directed_rounding_brackets_and_is_adjacent():
    rng = np.random.default_rng(4)
    for v in _sample_values(rng, 5000):
        if abs(v) > 65504:
            continue
        lo, hi = oracle.f16_rd(v), oracle.f16_ru(v)
        assert lo <= v <= hi
        assert float(np.float16(lo)) == lo and float(np.float16(hi)) == hi
        if lo != hi:
            assert float(np.nextafter(np.float16(lo), np.float16(np.inf))) == hi
        else:
            assert lo == v


def test_f16_bits_match_numpy_bit_patterns():
    pats = np.arange(0, 1 << 16, 7, dtype=np.uint16)
    vals = pats.view(np.float16).astype(np.float64)
    for p, v in zip(pats, vals):
        if np.isnan(v):
            continue
        assert oracle.f16_value(int(p)) == v
        assert oracle.f16_bits(v) == int(p)


def test_bf16_values_match_torch():
    x = torch.randn(1000, dtype=torch.float32) * 100
    b = x.to(torch.bfloat16)
    pats = b.view(torch.int16).numpy().astype(np.uint16)
    got = oracle.bf16_array_to_f64(pats)
    np.testing.assert_array_equal(got, b.to(torch.float64).numpy())
    for p, v in zip(pats[:50], got[:50]):
        assert oracle.bf16_value(int(p)) == v


# ---------------------------------------------------------------- VarN

def _block(seed, B, sigma_m=1.5, n_out=4, factor=20.0):
    g = synth.make_gen(seed)
    return synth.kv_values(g, 1, 1, B, sigma_m, n_out, factor)[0, 0].double().numpy()


@pytest.mark.parametrize("B,iters", [(32, 3), (64, 2), (32, 1), (64, 4)])
def test_varn_rows_then_columns_reach_unit_variance(B, iters):
    sb = synth.sign_bits(5)
    Xr = oracle.rotate(_block(B + iters, B), sb)
    Y, R, C, tr = oracle.varn(Xr, iters)
    # the last pass is the column pass: every column has population variance 1
    np.testing.assert_allclose(Y.var(axis=0), 1.0, atol=1e-12)
    # Y is Xr with rows divided by R and columns by C
    np.testing.assert_allclose(Y * R[:, None] * C[None, :], Xr, rtol=1e-12,
                               atol=1e-12 * np.abs(Xr).max())
    # the oracle's own trace: rows exactly 1 after each row pass, columns after each column pass
    assert np.all(tr[:, 0] < 1e-12) and np.all(tr[:, 1] < 1e-12)
    if iters == 1:
        # one pass each: independent numpy recomputation of the row pass
        rv = Xr.var(axis=1)
        np.testing.assert_allclose(R, np.sqrt(rv), rtol=1e-14)


def test_varn_row_variance_gap_shrinks_with_iterations():
    sb = synth.sign_bits(6)
    for seed in range(4):
        Xr = oracle.rotate(_block(100 + seed, 32), sb)
        _, _, _, tr = oracle.varn(Xr, 4)
        gap = tr[:, 2]
        assert np.all(np.diff(gap) <= 1e-15), gap   # Sinkhorn-type convergence
        assert gap[-1] < gap[0]


def test_varn_is_scale_equivariant_per_token():
    # the token pass runs first, so a token scaled by 2^k is normalised back
    # exactly and only its own factor moves
    sb = synth.sign_bits(8)
    X = _block(9, 32)
    base = oracle.quantize_block(X, 3, oracle.KIND_K, sb)
    X2 = X.copy()
    X2[5] *= 8.0                                    # exact power-of-two scaling of a token
    sc = oracle.quantize_block(X2, 3, oracle.KIND_K, sb)
    assert sc["R16"][5] == 8.0 * base["R16"][5]
    np.testing.assert_array_equal(np.delete(sc["R16"], 5), np.delete(base["R16"], 5))
    np.testing.assert_array_equal(sc["C16"], base["C16"])
    np.testing.assert_array_equal(sc["codes"], base["codes"])
    np.testing.assert_array_equal(sc["bytes"][:1024], base["bytes"][:1024])


def test_varn_degenerate_rows_and_columns_keep_factor_one():
    Xr = np.zeros((32, D))
    Y, R, C, _ = oracle.varn(Xr, 3)
    assert np.all(R == 1.0) and np.all(C == 1.0) and np.all(Y == 0.0)
    r = oracle.quantize_block(np.zeros((32, D)), 3, oracle.KIND_V, synth.sign_bits(1))
    assert np.all(r["codes"] == 0) and np.all(r["s16"] == 0) and np.all(r["z16"] == 0)
    dec = oracle.decode_blocks(r["bytes"], 32, oracle.KIND_V, synth.sign_bits(1), rotated=False)
    assert np.all(dec == 0.0)
    # identical tokens: after the token pass every channel is constant, so the
    # channel factors stay 1 and every token reconstructs to the same row
    row = np.random.default_rng(3).standard_normal(D)
    r = oracle.quantize_block(np.tile(row, (32, 1)), 3, oracle.KIND_K, synth.sign_bits(2))
    assert np.all(r["C"] == 1.0) and np.all(r["R"] == r["R"][0])
    dec = oracle.decode_blocks(r["bytes"], 32, oracle.KIND_K, synth.sign_bits(2), rotated=False)[0]
    assert np.all(dec == dec[0])


@pytest.mark.parametrize("mu", [1.0, -1.0, 4.0])
def test_varn_variance_threshold_is_two_sided(mu):
    # Reading R-5: a row or column is normalised only when its population
    # variance v exceeds 2^-30 * mu^2 (mu its mean). A line of alternating
    # mu + d, mu - d has mean mu and variance d^2 exactly in fp64, so the
    # factor is |d| just above the threshold and stays 1 at and below it.
    thr_d = 2.0 ** -15 * abs(mu)                 # d^2 = 2^-30 mu^2
    cases = [(thr_d * (1 + 2.0 ** -11), thr_d * (1 + 2.0 ** -11)),   # just above: factor d
             (thr_d, 1.0),                                         # at the threshold: kept
             (thr_d * (1 - 2.0 ** -11), 1.0)]                      # just below: kept
    rng = np.random.default_rng(21)
    for d, want in cases:
        alt = np.where(np.arange(D) % 2 == 0, mu + d, mu - d)
        Xr = rng.standard_normal((32, D))
        Xr[0] = alt
        _, R, _, _ = oracle.varn(Xr, 1, flags=oracle.NO_CHANNEL_PASS)
        assert R[0] == want, (mu, d, R[0])
        assert np.all(R[1:] != 1.0)                # the ordinary rows are normalised
        Xc = rng.standard_normal((32, D))
        Xc[:, 5] = np.where(np.arange(32) % 2 == 0, mu + d, mu - d)
        _, _, C, _ = oracle.varn(Xc, 1, flags=oracle.NO_TOKEN_PASS)
        assert C[5] == want, (mu, d, C[5])
    # the mean enters squared: at mu = 4 a variance 4 x 2^-30 (above 2^-30 mu
    # but below 2^-30 mu^2) keeps the factor
    if mu == 4.0:
        d = 2.0 ** -14
        Xr = rng.standard_normal((32, D))
        Xr[0] = np.where(np.arange(D) % 2 == 0, mu + d, mu - d)
        _, R, _, _ = oracle.varn(Xr, 1, flags=oracle.NO_CHANNEL_PASS)
        assert R[0] == 1.0


def test_round_factor_clamps_to_fp16_normal_range():
    assert oracle.round_factor(1e-9) == 2.0 ** -14
    assert oracle.round_factor(1e9) == 65504.0
    assert oracle.round_factor(1.0 + 2.0 ** -12) == 1.0
    assert oracle.round_factor(1.0 + 3 * 2.0 ** -12) == 1.0 + 2.0 ** -10


# ---------------------------------------------------------------- quantiser

def _all_f16_nonneg():
    pats = np.arange(0, 0x7C00, dtype=np.uint16)
    return pats.view(np.float16).astype(np.float64)


def test_group_params_are_the_brute_force_extremes():
    grid = _all_f16_nonneg()
    full = np.concatenate([-grid[::-1], grid])
    rng = np.random.default_rng(12)
    for _ in range(60):
        y = rng.standard_normal(32) * np.exp(rng.uniform(-6, 6)) + rng.uniform(-3, 3)
        z, s, m, M = oracle.group_params(y)
        assert m == y.min() and M == y.max()
        assert z == full[full <= m].max()                # largest fp16 <= min
        ok = grid[z + 3.0 * grid >= M]
        assert s == ok.min()                              # smallest fp16 covering the max


def test_step_rule_is_the_brute_force_minimum():
    grid = _all_f16_nonneg()
    rng = np.random.default_rng(15)
    for _ in range(200):
        z = float(np.float16(rng.uniform(-50, 50)))
        M = z + abs(rng.standard_normal()) * np.exp(rng.uniform(-12, 8))
        s = oracle.step_for(z, M)
        ok = grid[z + 3.0 * grid >= M]
        assert s == (ok.min() if ok.size else 65504.0)
    assert oracle.step_for(1.0, 1.0) == 0.0 and oracle.step_for(2.0, 1.0) == 0.0


def test_codes_are_nearest_levels_with_ties_to_even_and_error_at_most_half_step():
    sb = synth.sign_bits(2)
    for seed in range(3):
        X = _block(20 + seed, 64)
        r = oracle.quantize_block(X, 2, oracle.KIND_V, sb)
        y, z, s, codes = r["y"], r["z16"], r["s16"], r["codes"]
        for g in range(4):
            sl = slice(32 * g, 32 * g + 32)
            zz, ss = z[:, g:g + 1], s[:, g:g + 1]
            levels = zz[..., None] + ss[..., None] * np.arange(4)   # [B][1][4]
            dist = np.abs(y[:, sl][..., None] - levels)
            best = dist.min(axis=-1, keepdims=True)
            cand = np.where(dist == best, np.arange(4), 99)
            # argmin; exact ties go to the even level
            even = np.where((cand % 2 == 0) & (cand < 99), cand, 99).min(axis=-1)
            want = np.where((dist == best).sum(-1) > 1, even, cand.min(axis=-1))
            assert np.array_equal(codes[:, sl], want)
            yhat = zz + ss * codes[:, sl]
            assert np.all(np.abs(y[:, sl] - yhat) <= ss / 2 * (1 + 1e-15))
            # the group minimum always gets code 0
            assert np.all(codes[:, sl][np.arange(len(y)), y[:, sl].argmin(axis=1)] == 0)


def test_dequantised_block_is_within_half_step_of_the_input():
    sb = synth.sign_bits(4)
    X = _block(31, 32)
    for kind in (oracle.KIND_K, oracle.KIND_V):
        r = oracle.quantize_block(X, 3, kind, sb)
        rot = oracle.decode_blocks(r["bytes"], 32, kind, sb, rotated=True)[0]
        bound = (r["s16"].repeat(32, axis=1) / 2) * r["R16"][:, None] * r["C16"][None, :]
        assert np.all(np.abs(rot - r["Xr"]) <= bound * (1 + 1e-9) + 1e-300)
        unrot = oracle.decode_blocks(r["bytes"], 32, kind, sb, rotated=False)[0]
        err = np.linalg.norm(unrot - X, axis=1)
        assert np.all(err <= np.linalg.norm(bound, axis=1) * (1 + 1e-9))


def test_quantisation_is_local_to_the_head_block():
    sb = synth.sign_bits(5)
    A, Bk = _block(40, 32), _block(41, 32)
    two = oracle.quantize_blocks(np.stack([A, Bk]), 3, oracle.KIND_K, sb)
    other = oracle.quantize_blocks(np.stack([A, Bk * 3.0 + 1.0]), 3, oracle.KIND_K, sb)
    assert np.array_equal(two[0], other[0])
    assert np.array_equal(two[0], oracle.quantize_block(A, 3, oracle.KIND_K, sb)["bytes"])


# ---------------------------------------------------------------- packing

def _golden():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or ":" not in line:
            continue
        k, v = line.split(":", 1)
        out[k.strip()] = v.strip()
    return out


def test_pack_matches_hand_derived_bytes():
    gold = _golden()
    B = 32
    codes = np.tile(np.arange(D) % 4, (B, 1))
    s = np.ones((B, 4))
    z = -2.0 * np.ones((B, 4))
    R = 0.5 * np.ones(B)
    C = 2.0 * np.ones(D)
    kb = oracle.pack(B, oracle.KIND_K, codes, s, z, R, C)
    vb = oracle.pack(B, oracle.KIND_V, codes, s, z, R, C)
    assert kb[:32].tobytes().hex(" ") == gold["K c%4 first32"]
    assert vb[:32].tobytes().hex(" ") == gold["V c%4 first32"]
    assert kb[:1024].tobytes() == bytes.fromhex(gold["K c%4 first32"].replace(" ", "")) * 32
    assert vb[:1024].tobytes() == bytes.fromhex(gold["V c%4 first32"].replace(" ", "")) * 32
    offs = dict(zip(*[iter(gold["section offsets B=32"].split())] * 2))
    assert kb[int(offs["s"]):int(offs["s"]) + 2].tobytes().hex(" ") == gold["s bytes"]
    assert kb[int(offs["z"]):int(offs["z"]) + 2].tobytes().hex(" ") == gold["z bytes"]
    assert kb[int(offs["R"]):int(offs["R"]) + 2].tobytes().hex(" ") == gold["R bytes"]
    assert kb[int(offs["C"]):int(offs["C"]) + 2].tobytes().hex(" ") == gold["C bytes"]
    assert len(kb) == int(offs["total"]) == oracle.head_block_bytes(32)
    offs64 = dict(zip(*[iter(gold["section offsets B=64"].split())] * 2))
    assert oracle.head_block_bytes(64) == int(offs64["total"])
    all3 = oracle.pack(B, oracle.KIND_V, np.full((B, D), 3), s, z, R, C)
    assert set(all3[:1024].tolist()) == {int(gold["all3 code byte"], 16)}


def test_code_positions_are_a_bijection_and_pack_round_trips():
    for B in (32, 64):
        for kind in (0, 1):
            seen = set()
            for t in range(B):
                for c in range(D):
                    seen.add(oracle.code_position(kind, t, c))
            assert len(seen) == B * D
            assert all(b % 2 == 0 and 0 <= b < 32 for _, b in seen)
            rng = np.random.default_rng(B + kind)
            codes = rng.integers(0, 4, (B, D))
            f16 = lambda a: a.astype(np.float16).astype(np.float64)
            s, z = f16(np.abs(rng.standard_normal((B, 4)))), f16(rng.standard_normal((B, 4)))
            R, C = f16(np.abs(rng.standard_normal(B)) + 1), f16(np.abs(rng.standard_normal(D)) + 1)
            f = oracle.unpack(B, kind, oracle.pack(B, kind, codes, s, z, R, C))
            assert np.array_equal(f["codes"], codes)
            assert np.array_equal(f["s16"], s) and np.array_equal(f["z16"], z)
            assert np.array_equal(f["R16"], R) and np.array_equal(f["C16"], C)


# ---------------------------------------------------------------- attention

def test_rotated_query_route_equals_plain_attention():
    rng = np.random.default_rng(13)
    sb = synth.sign_bits(9)
    K = rng.standard_normal((40, D)) * np.exp(rng.standard_normal((40, 1)))
    V = rng.standard_normal((40, D)) * 3
    q = rng.standard_normal(D)
    a = oracle.attention(q, K, V, 1 / math.sqrt(D))
    b = oracle.attention_rotated(q, K, V, 1 / math.sqrt(D), sb)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-10)


def test_attention_closed_forms():
    rng = np.random.default_rng(14)
    V = rng.standard_normal((9, D))
    K = np.tile(rng.standard_normal(D), (9, 1))          # equal keys -> uniform weights
    q = rng.standard_normal(D)
    np.testing.assert_allclose(oracle.attention(q, K, V, 0.3), V.mean(0), atol=1e-13)
    K2 = rng.standard_normal((9, D))
    np.testing.assert_allclose(oracle.attention(np.zeros(D), K2, V, 0.3), V.mean(0), atol=1e-13)
    np.testing.assert_allclose(oracle.attention(q, K2[:1], V[:1], 0.3), V[0], atol=1e-15)
    # two keys: p1 = 1 / (1 + exp(l2 - l1))
    l = 0.3 * (K2[:2] @ q)
    p1 = 1.0 / (1.0 + math.exp(l[1] - l[0]))
    np.testing.assert_allclose(oracle.attention(q, K2[:2], V[:2], 0.3),
                               p1 * V[0] + (1 - p1) * V[1], atol=1e-12)


def test_decode_attention_pages_and_tail():
    """Paged, permuted blocks plus a bf16 tail equal attention over the
    concatenated decoded keys (assembled here with numpy indexing)."""
    B, n_q, n_kv, batch = 32, 4, 2, 3
    sb = synth.sign_bits(21)
    g = synth.make_gen(21)
    lens = [70, 32, 17]
    max_blocks = 3
    X = synth.kv_values(g, batch, n_kv, 96, 1.0, 2, 10.0)            # K
    Y = synth.kv_values(g, batch, n_kv, 96, 1.0, 2, 10.0)            # V
    Xb = X.to(torch.bfloat16)
    Yb = Y.to(torch.bfloat16)
    q = synth.queries(g, batch, n_q).double().numpy()
    perm = np.random.default_rng(0).permutation(batch * max_blocks).astype(np.int32)
    bt = perm.reshape(batch, max_blocks)
    hb = oracle.head_block_bytes(B)
    pool = np.zeros((batch * max_blocks, n_kv, 2, hb), dtype=np.uint8)
    staging = np.zeros((batch, n_kv, 2, B, D), dtype=np.uint16)
    for b in range(batch):
        for h in range(n_kv):
            for j in range(lens[b] // B):
                for kind, T in ((0, Xb), (1, Yb)):
                    vals = T[b, h, j * B:(j + 1) * B].double().numpy()
                    pool[bt[b, j], h, kind] = oracle.quantize_blocks(vals[None], 3, kind, sb)[0]
            tail = lens[b] % B
            base = (lens[b] // B) * B
            for kind, T in ((0, Xb), (1, Yb)):
                staging[b, h, kind, :tail] = T[b, h, base:base + tail].view(torch.int16).numpy()
    out = oracle.decode_attention(B, n_q, n_kv, sb, 1 / math.sqrt(D), q, pool, staging, bt,
                                  np.array(lens, dtype=np.int32))
    G = n_q // n_kv
    for b in range(batch):
        for h in range(n_kv):
            keys, vals = [], []
            nfull = lens[b] // B
            for j in range(nfull):
                keys.append(oracle.decode_blocks(pool[bt[b, j], h, 0], B, 0, sb, False)[0])
                vals.append(oracle.decode_blocks(pool[bt[b, j], h, 1], B, 1, sb, False)[0])
            tail = lens[b] % B
            keys.append(Xb[b, h, nfull * B:nfull * B + tail].double().numpy())
            vals.append(Yb[b, h, nfull * B:nfull * B + tail].double().numpy())
            Kc, Vc = np.concatenate(keys), np.concatenate(vals)
            for j in range(G):
                want = oracle.attention(q[b, h * G + j], Kc, Vc, 1 / math.sqrt(D))
                np.testing.assert_allclose(out[b, h * G + j], want, atol=1e-12)


# ---------------------------------------------------------------- ablation switches

def _largest_f16_at_most(m):
    h = np.float16(m)
    if float(h) > m:
        h = np.nextafter(h, np.float16(-np.inf))
    return float(h)


def test_no_rotation_no_varn_is_plain_group_quantisation():
    """With the rotation switched off and 0 VarN iterations the block is plain
    asymmetric 2-bit group quantisation of the raw values (R = C = 1)."""
    X = _block(70, 32)
    r = oracle.quantize_block(X, 0, oracle.KIND_K, [0, 0, 0, 0], flags=oracle.NO_ROTATION)
    assert np.array_equal(r["Xr"], X) and np.array_equal(r["y"], X)
    assert np.all(r["R16"] == 1.0) and np.all(r["C16"] == 1.0)
    for t in range(32):
        for g in range(4):
            grp = X[t, 32 * g:32 * g + 32]
            assert r["z16"][t, g] == _largest_f16_at_most(grp.min())
            # nearest of the four levels (exact ties never occur on this data)
            lv = r["z16"][t, g] + r["s16"][t, g] * np.arange(4)
            want = np.abs(grp[:, None] - lv[None, :]).argmin(axis=1)
            assert np.array_equal(r["codes"][t, 32 * g:32 * g + 32], want)
    # decoding never rotates back: both spaces coincide
    a = oracle.decode_blocks(r["bytes"], 32, 0, [0, 0, 0, 0], rotated=True, flags=oracle.NO_ROTATION)
    b = oracle.decode_blocks(r["bytes"], 32, 0, [0, 0, 0, 0], rotated=False, flags=oracle.NO_ROTATION)
    assert np.array_equal(a, b)
    assert np.all(np.abs(b[0] - X) <= r["s16"].repeat(32, axis=1) / 2 * (1 + 1e-15))


def test_hadamard_only_keeps_unit_factors():
    sb = synth.sign_bits(71)
    X = _block(71, 64)
    r = oracle.quantize_block(X, 0, oracle.KIND_V, sb)
    np.testing.assert_allclose(r["Xr"], oracle.rotate(X, sb), rtol=0, atol=0)
    assert np.all(r["R"] == 1.0) and np.all(r["C"] == 1.0)
    assert np.array_equal(r["y"], r["Xr"])


@pytest.mark.parametrize("iters", [1, 3])
def test_token_only_varn_is_the_row_spread(iters):
    """Channel pass off: C stays 1 and each R_t is the population standard
    deviation of its rotated row (repeating the pass changes nothing)."""
    sb = synth.sign_bits(72)
    X = _block(72, 32)
    r = oracle.quantize_block(X, iters, oracle.KIND_K, sb, flags=oracle.NO_CHANNEL_PASS)
    assert np.all(r["C"] == 1.0)
    np.testing.assert_allclose(r["R"], r["Xr"].std(axis=1), rtol=1e-12)


@pytest.mark.parametrize("iters", [1, 3])
def test_channel_only_varn_is_the_column_spread(iters):
    sb = synth.sign_bits(73)
    X = _block(73, 64)
    r = oracle.quantize_block(X, iters, oracle.KIND_K, sb, flags=oracle.NO_TOKEN_PASS)
    assert np.all(r["R"] == 1.0)
    np.testing.assert_allclose(r["C"], r["Xr"].std(axis=0), rtol=1e-12)


def test_varn_without_rotation_normalises_the_raw_block():
    """Rotation off, both passes on: the factors restore the raw block and the
    last (channel) pass leaves unit column variances."""
    X = _block(74, 32)
    Y, R, C, _ = oracle.varn(X, 3, oracle.NO_ROTATION)
    np.testing.assert_allclose(Y * R[:, None] * C[None, :], X, rtol=1e-12)
    np.testing.assert_allclose(Y.var(axis=0), 1.0, rtol=1e-12)
    r = oracle.quantize_block(X, 3, oracle.KIND_K, synth.sign_bits(74), flags=oracle.NO_ROTATION)
    assert np.array_equal(r["Xr"], X)
    np.testing.assert_allclose(r["R"], R, rtol=0)


def test_decode_attention_without_rotation_equals_plain_attention_over_decoded_keys():
    B, n_q, n_kv = 32, 4, 1
    sb = synth.sign_bits(75)
    g = synth.make_gen(75)
    K = synth.kv_values(g, 1, 1, 2 * B, 1.0, 2, 10.0)[0, 0].double().numpy()
    V = synth.kv_values(g, 1, 1, 2 * B, 1.0, 2, 10.0)[0, 0].double().numpy()
    q = synth.queries(g, 1, n_q).double().numpy()
    hb = oracle.head_block_bytes(B)
    pool = np.zeros((2, 1, 2, hb), dtype=np.uint8)
    f = oracle.NO_ROTATION | oracle.NO_CHANNEL_PASS
    for j in range(2):
        pool[j, 0, 0] = oracle.quantize_blocks(K[None, j * B:(j + 1) * B], 2, 0, sb, flags=f)[0]
        pool[j, 0, 1] = oracle.quantize_blocks(V[None, j * B:(j + 1) * B], 2, 1, sb, flags=f)[0]
    out = oracle.decode_attention(B, n_q, n_kv, sb, 0.1, q, pool, np.zeros((1, 1, 2, B, D), np.uint16),
                                  np.array([[1, 0]], np.int32), np.array([2 * B], np.int32), flags=f)
    Kd = np.concatenate([oracle.decode_blocks(pool[j, 0, 0], B, 0, sb, False, flags=f)[0] for j in (1, 0)])
    Vd = np.concatenate([oracle.decode_blocks(pool[j, 0, 1], B, 1, sb, False, flags=f)[0] for j in (1, 0)])
    for h in range(n_q):
        s = 0.1 * Kd @ q[0, h]
        p = np.exp(s - s.max())
        np.testing.assert_allclose(out[0, h], p @ Vd / p.sum(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- error decomposition

def test_error_split_closed_forms():
    """Magnitude / direction split of the quantisation error on vectors whose
    answer is known by hand."""
    rng = np.random.default_rng(80)
    x = rng.standard_normal(D)
    n = np.linalg.norm(x)
    np.testing.assert_allclose(oracle.error_split(x, x), [n, n, 0, 0], atol=1e-12)
    # pure scaling is all magnitude error: |E_M| = |k - 1| |x|
    np.testing.assert_allclose(oracle.error_split(x, 2.5 * x), [n, 2.5 * n, 1.5 * n, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.error_split(x, 0.25 * x), [n, 0.25 * n, 0.75 * n, 0], rtol=1e-12,
                               atol=1e-12)
    # a rotation by 90 degrees at equal length is all direction error: |E_D| = sqrt(2) |x|
    e = np.zeros(D); e[3] = 2.0
    f = np.zeros(D); f[17] = 2.0
    np.testing.assert_allclose(oracle.error_split(e, f), [2, 2, 0, 2 * math.sqrt(2)], rtol=1e-12)
    # opposite direction, 3x the length: |E_M| = 2|x|, |E_D| = 3|x| * 2
    np.testing.assert_allclose(oracle.error_split(e, -3 * e), [2, 6, 4, 12], rtol=1e-12)
    # the degenerate ends of the reading
    np.testing.assert_allclose(oracle.error_split(np.zeros(D), f), [0, 2, 2, 0])
    np.testing.assert_allclose(oracle.error_split(e, np.zeros(D)), [2, 0, 2, 0])


def test_error_split_parts_add_up_to_the_error():
    """|E_M + E_D| = |x^ - x| and the triangle inequality, on quantised data."""
    sb = synth.sign_bits(81)
    X = _block(81, 32)
    r = oracle.quantize_block(X, 3, oracle.KIND_K, sb)
    Xh = oracle.decode_blocks(r["bytes"], 32, 0, sb, rotated=False)[0]
    out = oracle.error_decomposition(X[None], r["bytes"][None], 32, 0, sb)[0]
    for t in range(32):
        nx, nh, em, ed = out[t]
        assert nx == pytest.approx(np.linalg.norm(X[t]), rel=1e-12)
        assert nh == pytest.approx(np.linalg.norm(Xh[t]), rel=1e-12)
        err = np.linalg.norm(Xh[t] - X[t])
        # E_M is parallel to x and E_D = x^ - |x^| x/|x|, so |E_M + E_D|^2 follows from
        # the law of cosines on x^ and x: both sides computed independently here
        cos = X[t] @ Xh[t] / (nx * nh)
        assert ed == pytest.approx(nh * math.sqrt(max(0.0, 2 - 2 * cos)), rel=1e-6, abs=1e-12)
        assert em <= err * (1 + 1e-12) and ed <= err + em + 1e-12 and err <= em + ed + 1e-12


# ---------------------------------------------------------------- 4-bit width

def test_pack_4bit_matches_hand_derived_bytes():
    gold = _golden()
    B = 32
    s, z = np.ones((B, 4)), -2.0 * np.ones((B, 4))
    R, C = 0.5 * np.ones(B), 2.0 * np.ones(D)
    kcodes = np.tile(np.arange(D) % 16, (B, 1))
    vcodes = np.tile((np.arange(B) % 16)[:, None], (1, D))
    kb = oracle.pack(B, oracle.KIND_K, kcodes, s, z, R, C, bits=4)
    vb = oracle.pack(B, oracle.KIND_V, vcodes, s, z, R, C, bits=4)
    for key, buf in (("K4 c%16", kb), ("V4 t%16", vb)):
        w0 = bytes.fromhex(gold[f"{key} record0 word"].replace(" ", ""))
        w1 = bytes.fromhex(gold[f"{key} record1 word"].replace(" ", ""))
        assert buf[:64].tobytes() == w0 * 16 and buf[64:128].tobytes() == w1 * 16
    offs = dict(zip(*[iter(gold["section offsets 4-bit B=32"].split())] * 2))
    assert kb[int(offs["s"]):int(offs["s"]) + 2].tobytes().hex(" ") == gold["s bytes"]
    assert kb[int(offs["C"]):int(offs["C"]) + 2].tobytes().hex(" ") == gold["C bytes"]
    assert len(kb) == int(offs["total"]) == oracle.head_block_bytes(32, 4)
    offs64 = dict(zip(*[iter(gold["section offsets 4-bit B=64"].split())] * 2))
    assert oracle.head_block_bytes(64, 4) == int(offs64["total"])


def test_4bit_positions_are_a_bijection_and_pack_round_trips():
    for B in (32, 64):
        for kind in (0, 1):
            seen = {oracle.code_position(kind, t, c, bits=4) for t in range(B) for c in range(D)}
            assert len(seen) == B * D
            assert all(b % 4 == 0 and 0 <= b < 32 for _, b in seen)
            assert max(w for w, _ in seen) == 4 * B * 4 - 1
            rng = np.random.default_rng(40 + B + kind)
            codes = rng.integers(0, 16, (B, D))
            f16 = lambda a: a.astype(np.float16).astype(np.float64)
            s, z = f16(np.abs(rng.standard_normal((B, 4)))), f16(rng.standard_normal((B, 4)))
            R, C = f16(np.abs(rng.standard_normal(B)) + 1), f16(np.abs(rng.standard_normal(D)) + 1)
            f = oracle.unpack(B, kind, oracle.pack(B, kind, codes, s, z, R, C, bits=4), bits=4)
            assert np.array_equal(f["codes"], codes)
            assert np.array_equal(f["s16"], s) and np.array_equal(f["R16"], R) and np.array_equal(f["C16"], C)


def test_4bit_group_params_and_codes_are_brute_force():
    grid = _all_f16_nonneg()
    full = np.concatenate([-grid[::-1], grid])
    rng = np.random.default_rng(41)
    for _ in range(40):
        y = rng.standard_normal(32) * np.exp(rng.uniform(-6, 6)) + rng.uniform(-3, 3)
        z, s, m, M = oracle.group_params(y, bits=4)
        assert z == full[full <= m].max()
        assert s == grid[z + 15.0 * grid >= M].min()          # 15 steps cover the group
        lv = z + s * np.arange(16)
        for v in y:
            d = np.abs(v - lv)
            want = np.flatnonzero(d == d.min())
            want = want[0] if len(want) == 1 else [k for k in want if k % 2 == 0][0]
            assert oracle.code(v, z, s, bits=4) == want
            assert abs(v - lv[oracle.code(v, z, s, bits=4)]) <= s / 2 * (1 + 1e-15)


def test_4bit_block_is_within_half_step_and_finer_than_2bit():
    sb = synth.sign_bits(42)
    X = _block(42, 64)
    errs = {}
    for bits in (2, 4):
        r = oracle.quantize_block(X, 2, oracle.KIND_K, sb, bits=bits)
        rot = oracle.decode_blocks(r["bytes"], 64, 0, sb, rotated=True, bits=bits)[0]
        bound = (r["s16"].repeat(32, axis=1) / 2) * r["R16"][:, None] * r["C16"][None, :]
        assert np.all(np.abs(rot - r["Xr"]) <= bound * (1 + 1e-9) + 1e-300)
        assert r["codes"].max() <= (1 << bits) - 1
        unrot = oracle.decode_blocks(r["bytes"], 64, 0, sb, rotated=False, bits=bits)[0]
        errs[bits] = np.linalg.norm(unrot - X) / np.linalg.norm(X)
    # the same factors, 15 steps per group instead of 3: roughly 5x finer
    assert errs[4] < errs[2] / 3


# ---------------------------------------------------------------- chunked prefill attention

def _paged_cache(B, n_kv, batch, lens, max_blocks, K, V, sb, iters=3, bits=2):
    """Pool (permuted blocks) and staging holding K, V ([batch][n_kv][L][128]
    bf16 tensors) for the given lengths, built with the oracle's quantiser."""
    perm = np.random.default_rng(batch + max_blocks).permutation(batch * max_blocks).astype(np.int32)
    bt = perm.reshape(batch, max_blocks)
    hb = oracle.head_block_bytes(B, bits)
    pool = np.zeros((batch * max_blocks, n_kv, 2, hb), dtype=np.uint8)
    staging = np.zeros((batch, n_kv, 2, B, D), dtype=np.uint16)
    for b in range(batch):
        for h in range(n_kv):
            nfull = lens[b] // B
            for kind, T in ((0, K), (1, V)):
                for j in range(nfull):
                    vals = T[b, h, j * B:(j + 1) * B].double().numpy()
                    pool[bt[b, j], h, kind] = oracle.quantize_blocks(vals[None], iters, kind, sb, bits=bits)[0]
                tail = lens[b] - nfull * B
                staging[b, h, kind, :tail] = T[b, h, nfull * B:lens[b]].view(torch.int16).numpy()
    return pool, staging, bt


def test_prefill_chunk_of_one_is_decode_attention():
    """A chunk of one query per sequence is the decode step over the same cache."""
    B, n_q, n_kv, batch = 32, 4, 2, 3
    sb = synth.sign_bits(90)
    g = synth.make_gen(90)
    lens = [70, 32, 17]
    K = synth.kv_values(g, batch, n_kv, 96, 1.0, 2, 10.0).to(torch.bfloat16)
    V = synth.kv_values(g, batch, n_kv, 96, 1.0, 2, 10.0).to(torch.bfloat16)
    q = synth.queries(g, batch, n_q).double().numpy()
    pool, staging, bt = _paged_cache(B, n_kv, batch, lens, 3, K, V, sb)
    sl = np.array(lens, np.int32)
    dec = oracle.decode_attention(B, n_q, n_kv, sb, 0.2, q, pool, staging, bt, sl)
    pre = oracle.prefill_attention(B, n_q, n_kv, sb, 0.2, q[:, None], pool, staging, bt, sl)
    assert np.array_equal(pre[:, 0], dec)


@pytest.mark.parametrize("bits", [2, 4])
def test_prefill_identical_keys_average_the_visible_values(bits):
    """All keys equal (zero keys: every score 0) -> each row is the plain mean
    of the values it may see: the first p + 1 tokens, decoded or raw."""
    B, n_q, n_kv, batch, chunk = 32, 2, 1, 2, 40
    sb = synth.sign_bits(91)
    g = synth.make_gen(91)
    lens = [75, 30]                      # the second has rows at negative positions
    K = torch.zeros(batch, n_kv, 96, D, dtype=torch.bfloat16)
    V = synth.kv_values(g, batch, n_kv, 96, 1.0, 2, 10.0).to(torch.bfloat16)
    pool, staging, bt = _paged_cache(B, n_kv, batch, lens, 3, K, V, sb, bits=bits)
    q = synth.queries(g, batch * chunk, n_q).double().numpy().reshape(batch, chunk, n_q, D)
    out = oracle.prefill_attention(B, n_q, n_kv, sb, 0.3, q, pool, staging, bt, np.array(lens, np.int32),
                                   bits=bits)
    for b in range(batch):
        nfull = lens[b] // B
        rows = [oracle.decode_blocks(pool[bt[b, j], 0, 1], B, 1, sb, False, bits=bits)[0] for j in range(nfull)]
        rows.append(V[b, 0, nfull * B:lens[b]].double().numpy())
        Vc = np.concatenate(rows)
        for r in range(chunk):
            p = lens[b] - chunk + r
            want = Vc[:p + 1].mean(axis=0) if p >= 0 else np.zeros(D)
            for h in range(n_q):
                np.testing.assert_allclose(out[b, r, h], want, rtol=1e-12, atol=1e-12)


def test_prefill_is_causal():
    """Changing the raw tail row of position p0 (K and V) leaves every row
    before p0 as it was and changes the rows at or after it (a small softmax
    scale keeps every visible token's weight well above zero)."""
    B, n_q, n_kv, batch, chunk = 32, 4, 2, 1, 24
    sb = synth.sign_bits(92)
    g = synth.make_gen(92)
    L = 2 * B + 20                       # 20 raw rows; the chunk spans a complete block and the tail
    K = synth.kv_values(g, batch, n_kv, L, 1.0, 2, 10.0).to(torch.bfloat16)
    V = synth.kv_values(g, batch, n_kv, L, 1.0, 2, 10.0).to(torch.bfloat16)
    pool, staging, bt = _paged_cache(B, n_kv, batch, [L], 3, K, V, sb)
    q = synth.queries(g, chunk, n_q).double().numpy().reshape(1, chunk, n_q, D)
    sl = np.array([L], np.int32)
    base = oracle.prefill_attention(B, n_q, n_kv, sb, 0.01, q, pool, staging, bt, sl)
    p0 = 2 * B + 10
    st2 = staging.copy()
    st2[0, :, :, p0 - 2 * B] = torch.full((n_kv, 2, D), 3.0, dtype=torch.bfloat16).view(torch.int16).numpy()
    moved = oracle.prefill_attention(B, n_q, n_kv, sb, 0.01, q, pool, st2, bt, sl)
    r0 = p0 - (L - chunk)
    assert np.array_equal(moved[0, :r0], base[0, :r0])
    assert np.all(np.abs(moved[0, r0:] - base[0, r0:]).max(axis=(1, 2)) > 1e-3)


# ---------------------------------------------------------------- 3-bit width (2-bit plane + 1-bit plane)

def test_pack_3bit_matches_hand_derived_bytes():
    gold = _golden()
    B = 32
    s, z = np.ones((B, 4)), -2.0 * np.ones((B, 4))
    R, C = 0.5 * np.ones(B), 2.0 * np.ones(D)
    kcodes = np.tile(np.arange(D) % 8, (B, 1))
    vcodes = np.tile((np.arange(B) % 8)[:, None], (1, D))
    kb = oracle.pack(B, oracle.KIND_K, kcodes, s, z, R, C, bits=3)
    vb = oracle.pack(B, oracle.KIND_V, vcodes, s, z, R, C, bits=3)
    for key, buf in (("K3 c%8", kb), ("V3 t%8", vb)):
        lo = bytes.fromhex(gold[f"{key} low word"].replace(" ", ""))
        hi = bytes.fromhex(gold[f"{key} high word"].replace(" ", ""))
        for rec in range(32):
            assert buf[48 * rec:48 * rec + 48].tobytes() == lo * 8 + hi * 4
    offs = dict(zip(*[iter(gold["section offsets 3-bit B=32"].split())] * 2))
    assert kb[int(offs["s"]):int(offs["s"]) + 2].tobytes().hex(" ") == gold["s bytes"]
    assert kb[int(offs["R"]):int(offs["R"]) + 2].tobytes().hex(" ") == gold["R bytes"]
    assert len(kb) == int(offs["total"]) == oracle.head_block_bytes(32, 3)
    offs64 = dict(zip(*[iter(gold["section offsets 3-bit B=64"].split())] * 2))
    assert oracle.head_block_bytes(64, 3) == int(offs64["total"])


def test_3bit_positions_cover_every_bit_once_and_pack_round_trips():
    for B in (32, 64):
        for kind in (0, 1):
            used = set()
            for t in range(B):
                for c in range(D):
                    w, b = oracle.code_position(kind, t, c, bits=3)
                    wh, bh = oracle.code_high_position(kind, t, c)
                    assert w % 12 < 8 and b % 2 == 0 and wh % 12 >= 8 and w // 12 == wh // 12
                    for bit in ((w, b), (w, b + 1), (wh, bh)):
                        assert bit not in used
                        used.add(bit)
            assert len(used) == 32 * 4 * B * 3          # every bit of the code section
            rng = np.random.default_rng(50 + B + kind)
            codes = rng.integers(0, 8, (B, D))
            f16 = lambda a: a.astype(np.float16).astype(np.float64)
            s, z = f16(np.abs(rng.standard_normal((B, 4)))), f16(rng.standard_normal((B, 4)))
            R, C = f16(np.abs(rng.standard_normal(B)) + 1), f16(np.abs(rng.standard_normal(D)) + 1)
            f = oracle.unpack(B, kind, oracle.pack(B, kind, codes, s, z, R, C, bits=3), bits=3)
            assert np.array_equal(f["codes"], codes)
            assert np.array_equal(f["z16"], z) and np.array_equal(f["C16"], C)


def test_3bit_group_params_and_codes_are_brute_force():
    grid = _all_f16_nonneg()
    full = np.concatenate([-grid[::-1], grid])
    rng = np.random.default_rng(51)
    for _ in range(40):
        y = rng.standard_normal(32) * np.exp(rng.uniform(-6, 6)) + rng.uniform(-3, 3)
        z, s, m, M = oracle.group_params(y, bits=3)
        assert z == full[full <= m].max()
        assert s == grid[z + 7.0 * grid >= M].min()           # 7 steps cover the group
        lv = z + s * np.arange(8)
        for v in y:
            d = np.abs(v - lv)
            want = np.flatnonzero(d == d.min())
            want = want[0] if len(want) == 1 else [k for k in want if k % 2 == 0][0]
            assert oracle.code(v, z, s, bits=3) == want


def test_3bit_block_is_within_half_step_between_2_and_4_bits():
    sb = synth.sign_bits(52)
    X = _block(52, 32)
    errs = {}
    for bits in (2, 3, 4):
        r = oracle.quantize_block(X, 3, oracle.KIND_V, sb, bits=bits)
        rot = oracle.decode_blocks(r["bytes"], 32, 1, sb, rotated=True, bits=bits)[0]
        bound = (r["s16"].repeat(32, axis=1) / 2) * r["R16"][:, None] * r["C16"][None, :]
        assert np.all(np.abs(rot - r["Xr"]) <= bound * (1 + 1e-9) + 1e-300)
        assert r["codes"].max() <= (1 << bits) - 1
        errs[bits] = np.linalg.norm(rot - r["Xr"])
    assert errs[4] < errs[3] < errs[2]
