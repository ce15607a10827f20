"""The staged parity check itself, on the CPU: it accepts the oracle's own
bytes with nothing excused, excuses only the neighbour across a nearby
rounding boundary, and rejects every other planted difference (a code off by
one away from a boundary, a code off by two, a zero or step one fp16 value
away from a grid point that is not near)."""
import numpy as np
import pytest

import oracle
import synth
from kvtest_util import code_flip_ok, staged_quantize_parity, step_window, zero_window

B = 32


def _block(seed):
    g = synth.make_gen(seed)
    return synth.kv_values(g, 1, 1, B, 1.5, 4, 20.0)[0, 0].double().numpy()


def _oracle_bytes(X, kind, sb):
    return oracle.quantize_block(X, 3, kind, sb)


def test_oracle_bytes_pass_with_nothing_excused():
    sb = synth.sign_bits(11)
    for kind in (oracle.KIND_K, oracle.KIND_V):
        X = _block(40 + kind)
        r = _oracle_bytes(X, kind, sb)
        st = staged_quantize_parity(X[None], r["bytes"][None], B, 3, kind, sb)
        assert st["codes"] == B * 128 and st["groups"] == B * 4
        assert st["factor_excused"] == st["zero_excused"] == st["step_excused"] == st["code_excused"] == 0


def _repack(r, kind, **over):
    f = dict(codes=r["codes"].copy(), s16=r["s16"].copy(), z16=r["z16"].copy(), R16=r["R16"], C16=r["C16"])
    for k, v in over.items():
        f[k] = v
    return oracle.pack(B, kind, f["codes"], f["s16"], f["z16"], f["R16"], f["C16"])


def test_planted_code_differences_fail():
    sb = synth.sign_bits(12)
    X = _block(50)
    r = _oracle_bytes(X, oracle.KIND_K, sb)
    y = oracle.normalise(r["Xr"], r["R16"], r["C16"])
    codes, dist = oracle.codes_given(y, r["z16"], r["s16"])
    # the code farthest from any boundary, moved to a neighbour
    t, c = np.unravel_index(np.argmax(np.where(np.isfinite(dist), dist, -1)), dist.shape)
    bad = r["codes"].copy()
    bad[t, c] = bad[t, c] + 1 if bad[t, c] < 3 else bad[t, c] - 1
    with pytest.raises(AssertionError, match="code mismatch"):
        staged_quantize_parity(X[None], _repack(r, oracle.KIND_K, codes=bad)[None], B, 3, oracle.KIND_K, sb)
    # a code moved by two, whatever its distance
    bad = r["codes"].copy()
    bad[t, c] = 2 if bad[t, c] < 2 else 0
    with pytest.raises(AssertionError, match="code mismatch"):
        staged_quantize_parity(X[None], _repack(r, oracle.KIND_K, codes=bad)[None], B, 3, oracle.KIND_K, sb)


def test_planted_zero_and_step_differences_fail():
    sb = synth.sign_bits(13)
    X = _block(60)
    r = _oracle_bytes(X, oracle.KIND_V, sb)
    z = r["z16"].copy()
    z[3, 1] = oracle.f16_rd(np.nextafter(z[3, 1], -np.inf))   # the fp16 value below the oracle's zero
    with pytest.raises(AssertionError, match="z16 mismatch"):
        staged_quantize_parity(X[None], _repack(r, oracle.KIND_V, z16=z)[None], B, 3, oracle.KIND_V, sb)
    s = r["s16"].copy()
    s[5, 2] = oracle.f16_ru(np.nextafter(s[5, 2], np.inf))    # the fp16 value above the oracle's step
    with pytest.raises(AssertionError, match="s16 mismatch"):
        staged_quantize_parity(X[None], _repack(r, oracle.KIND_V, s16=s)[None], B, 3, oracle.KIND_V, sb)


def test_zero_rule_allows_only_the_neighbour_across_a_near_grid_point():
    below_one = oracle.f16_rd(np.nextafter(1.0, 0.0))            # 1 - 2^-11
    assert below_one == 1.0 - 2.0 ** -11
    # a minimum on the grid point 1.0: either side of it is within the window
    assert zero_window(1.0, 2.0) == (below_one, 1.0)
    # a minimum a hair above the grid point: still both
    assert zero_window(1.0 + 1e-7, 2.0) == (below_one, 1.0)
    # a minimum half-way between two fp16 values: only the round-down
    assert zero_window(1.0 + 2.0 ** -11, 2.0) == (1.0, 1.0)
    # the window is relative to the group's range: a minimum near zero in a
    # group of range 1 may round to any fp16 value within 1e-5 of it
    lo, hi = zero_window(2.0 ** -20, 1.0)
    assert lo == oracle.f16_rd(2.0 ** -20 - 1e-5) < 0.0 < hi == oracle.f16_rd(2.0 ** -20 + 1e-5)


def test_step_rule_allows_only_the_neighbour_across_a_near_grid_point():
    # (M - z)/3 exactly 1.0: the covering step is 1.0; a maximum within the
    # window above needs the fp16 value above 1.0
    z, M = 0.0, 3.0
    assert step_window(z, M, 2) == (1.0, 1.0 + 2.0 ** -10)
    # half-way between grid points: one value only
    M2 = 3.0 * (1.0 + 2.0 ** -11)
    s2 = oracle.step_for(z, M2, bits=2)
    assert step_window(z, M2, 2) == (s2, s2) and s2 == 1.0 + 2.0 ** -10


def test_code_flip_rule():
    z, s = -1.5, 1.0
    b01 = z + 0.5 * s                     # boundary between codes 0 and 1
    assert code_flip_ok(b01 + 1e-9, z, s, 0, 1) and code_flip_ok(b01 - 1e-9, z, s, 1, 0)
    assert not code_flip_ok(b01 + 1e-3, z, s, 0, 1)   # far from the boundary
    assert not code_flip_ok(z + 1.5 * s, z, s, 0, 2)  # not neighbours
    assert not code_flip_ok(b01, z, s, 1, 2)           # neighbours, but not across this boundary
    assert not code_flip_ok(z, z, 0.0, 0, 1)           # a constant group has one level
