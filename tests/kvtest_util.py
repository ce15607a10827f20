"""Shared helpers for the KVarN tests: the staged quantiser parity check and
paged-cache construction on the GPU through the C ABI.

Parity rules (staged hand-off; each stage is recomputed from the GPU's
already-validated rounded values so one boundary case cannot cascade):
  factors  R16, C16 equal the oracle's fp16 rounding of its fp64 factors, or
           the oracle value lies within 1e-5 relative of the rounding midpoint
           between the two and the GPU value is one of those two (counted);
  z16/s16  recomputed by the oracle from its fp64 rotated values and the GPU's
           R16, C16: equal, or the GPU value is what the rounding rule gives
           for some pre-rounding value within 1e-5 of the oracle's, relative
           to the group's own scale: max(|m|, M - m) for the zero (group
           minimum m, maximum M), (M - z)/L for the step, L = 2^bits - 1
           (counted; so only the fp16 neighbour across a nearby grid point is
           excused, never a value further away);
  codes    recomputed from that y with the GPU's z16, s16: equal, or the GPU
           code is the oracle's +-1 and y lies within 1e-6 * max(1, |b|) of
           the decision boundary b between the two codes (counted; the count
           over a test's whole population must stay <= 1e-6 of its codes,
           checked by assert_code_flip_rate).
"""
from __future__ import annotations

import math
import os
from collections import Counter

import numpy as np
import torch

import oracle

D = 128


def f16_neighbours(v: float):
    lo, hi = oracle.f16_rd(v), oracle.f16_ru(v)
    return lo, hi


def zero_window(m: float, M: float):
    """The fp16 zeros the rule allows for a group with minimum m and maximum
    M, as a closed interval: the round-down of every value within
    1e-5 * max(|m|, M - m) of m (the clamp to the fp16 range applied first,
    as the oracle does). For a minimum of the group's own size the window is
    far below one fp16 spacing, so the interval holds the oracle's zero and
    at most the neighbour across a grid point inside the window."""
    eps = 1e-5 * max(abs(m), M - m)
    lo = min(max(m - eps, -65504.0), 65504.0)
    hi = min(max(m + eps, -65504.0), 65504.0)
    return oracle.f16_rd(lo), oracle.f16_rd(hi)


def step_window(z16: float, M: float, bits: int):
    """The fp16 steps the rule allows for zero z16 and group maximum M, as a
    closed interval: the least covering step for every maximum whose
    pre-rounding step (M - z)/L lies within 1e-5 relative of the oracle's
    (the rule is monotone in the maximum)."""
    d = 1e-5 * abs(M - z16)
    return oracle.step_for(z16, M - d, bits=bits), oracle.step_for(z16, M + d, bits=bits)


def in_window(v: float, w) -> bool:
    return w[0] <= v <= w[1]


def code_flip_ok(y: float, z16: float, s16: float, k_gpu: int, k_ref: int) -> bool:
    """An excusable code mismatch: the two codes are neighbours and y lies
    within 1e-6 * max(1, |b|) of the decision boundary b between them."""
    if abs(int(k_gpu) - int(k_ref)) != 1 or s16 <= 0.0:
        return False
    b = z16 + (min(int(k_gpu), int(k_ref)) + 0.5) * s16
    return abs(y - b) <= 1e-6 * max(1.0, abs(b))


def staged_quantize_parity(X: np.ndarray, gpu_bytes: np.ndarray, B: int, iters: int, kind: int,
                           sign_bits, flags: int = 0, bits: int = 2) -> Counter:
    """X: [n][B][128] float64 inputs exactly as the GPU read them; gpu_bytes:
    [n][head_block_bytes] uint8. Raises AssertionError on a violation."""
    st = Counter()
    X = np.asarray(X, dtype=np.float64)
    n = X.shape[0]
    for i in range(n):
        ref = oracle.quantize_block(X[i], iters, kind, sign_bits, flags=flags, bits=bits)
        f = oracle.unpack(B, kind, gpu_bytes[i], bits=bits)
        # ---- factors
        raw = np.concatenate([ref["R"], ref["C"]])
        got = np.concatenate([f["R16"], f["C16"]])
        want = np.concatenate([ref["R16"], ref["C16"]])
        bad = np.nonzero(got != want)[0]
        for k in bad:
            v = min(max(raw[k], 2.0 ** -14), 65504.0)
            lo, hi = f16_neighbours(v)
            mid = 0.5 * (lo + hi)
            ok = got[k] in (lo, hi) and want[k] in (lo, hi) and abs(v - mid) <= 1e-5 * v
            assert ok, f"block {i} factor {k}: gpu {got[k]!r} oracle {want[k]!r} (value {raw[k]!r})"
            st["factor_excused"] += 1
        st["factors"] += raw.size
        # ---- group zero and step from the GPU's factors
        y = oracle.normalise(ref["Xr"], f["R16"], f["C16"])
        z_o, _, m, M = oracle.group_params_all(y, bits=bits)
        zb = np.nonzero(f["z16"] != z_o)
        for t, g in zip(*zb):
            assert in_window(f["z16"][t, g], zero_window(m[t, g], M[t, g])), (
                f"block {i}: z16 mismatch gpu {f['z16'][t, g]!r} oracle {z_o[t, g]!r} "
                f"min {m[t, g]!r} max {M[t, g]!r}")
            st["zero_excused"] += 1
        s_o = np.array([[oracle.step_for(f["z16"][t, g], M[t, g], bits=bits) for g in range(4)]
                        for t in range(B)])
        sb_ = np.nonzero(f["s16"] != s_o)
        for t, g in zip(*sb_):
            assert in_window(f["s16"][t, g], step_window(f["z16"][t, g], M[t, g], bits)), (
                f"block {i}: s16 mismatch gpu {f['s16'][t, g]!r} oracle {s_o[t, g]!r} "
                f"zero {f['z16'][t, g]!r} max {M[t, g]!r}")
            st["step_excused"] += 1
        st["groups"] += B * 4
        # ---- codes from y with the GPU's z16, s16
        codes, dist = oracle.codes_given(y, f["z16"], f["s16"], bits=bits)
        cb = np.nonzero(codes != f["codes"])
        for t, c in zip(*cb):
            g = c // 32
            assert code_flip_ok(y[t, c], f["z16"][t, g], f["s16"][t, g], f["codes"][t, c], codes[t, c]), (
                f"block {i}: code mismatch at token {t} channel {c}: gpu {f['codes'][t, c]} oracle "
                f"{codes[t, c]} y {y[t, c]!r} zero {f['z16'][t, g]!r} step {f['s16'][t, g]!r}")
            st["code_excused"] += 1
        st["codes_in_window"] += int(np.sum(dist <= 1e-6 * np.maximum(1.0, np.abs(y))))
        st["codes"] += B * D
    return st


def assert_code_flip_rate(st: Counter, rate: float = 1e-6):
    """Excused code flips over a test's whole population stay <= rate."""
    assert st["code_excused"] <= rate * st["codes"] or st["code_excused"] == 0, dict(st)


def attn_close(got: np.ndarray, ref: np.ndarray, tol: float = 2e-3):
    """|got - ref| <= tol * max(1, |ref|) elementwise; returns the worst ratio."""
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    worst = float(np.nanmax(err)) if err.size else 0.0
    assert np.all(np.isfinite(got)), "non-finite attention output"
    assert worst <= tol, f"attention error {worst:.3e} > {tol}"
    log = os.environ.get("KVARN_ERROR_LOG")   # optional: one line per check, for margin reports
    if log:
        with open(log, "a") as f:
            f.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]} {worst:.4e}\n")
    return worst


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class PagedCache:
    """A packed paged cache (the config's code width) built through the C ABI.

    block_table[b][j] is a physical block id (a seeded permutation when
    perm_seed is given); staging holds the raw tail rows.
    """

    def __init__(self, kv, cfg, batch: int, max_blocks: int, perm_seed=None, device="cuda",
                 extra_blocks: int = 0):
        self.kv, self.cfg = kv, cfg
        self.B = cfg.block_size
        self.batch, self.max_blocks = batch, max_blocks
        n_pool = batch * max_blocks + extra_blocks
        ids = np.arange(batch * max_blocks, dtype=np.int32)
        if perm_seed is not None:
            ids = np.random.default_rng(perm_seed).permutation(batch * max_blocks).astype(np.int32)
        self.block_table_np = ids.reshape(batch, max_blocks)
        self.block_table = torch.from_numpy(self.block_table_np).to(device)
        self.pool = kv.alloc_pool(cfg, n_pool, device)
        self.staging = kv.alloc_staging(cfg, batch, device)
        self.ws = kv.alloc_workspace(cfg, 0, 0, device)
        self.hb = kv.head_block_bytes(cfg)
        self.bb = kv.block_bytes(cfg)

    def head_block_offset(self, b, h, j, kind):
        return int(self.block_table_np[b, j]) * self.bb + (2 * h + kind) * self.hb

    def prefill(self, K: torch.Tensor, V: torch.Tensor, lens):
        """K, V: bf16 or fp32 [batch][n_kv][Lmax][128] on the GPU."""
        B = self.B
        n_kv = self.cfg.n_kv_heads
        for b, L in enumerate(lens):
            nb = L // B
            for h in range(n_kv):
                for kind, T in ((0, K), (1, V)):
                    if nb > 0:
                        offs = torch.tensor([self.head_block_offset(b, h, j, kind) for j in range(nb)],
                                            dtype=torch.int64, device=T.device)
                        src = T[b, h, :nb * B].contiguous()
                        self.kv.quantize_block(self.cfg, kind, src, self.pool, self.ws, dst_offsets=offs,
                                               n_head_blocks=nb)
                    tail = L - nb * B
                    if tail > 0:
                        self.staging[b, h, kind, :tail] = T[b, h, nb * B:L].to(torch.bfloat16)
        torch.cuda.synchronize()

    def head_block(self, b, h, j, kind) -> np.ndarray:
        o = self.head_block_offset(b, h, j, kind)
        return self.pool.view(-1)[o:o + self.hb].cpu().numpy()


def oracle_attention(cache: PagedCache, q: torch.Tensor, seq_lens, sign_bits, sm_scale=None, seqs=None,
                     pool_np=None):
    """Oracle attention over the GPU's own cache bytes; seqs selects a sample
    of sequences (the result then has one row per selected sequence)."""
    cfg = cache.cfg
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    seqs = list(range(q.shape[0])) if seqs is None else list(seqs)
    qn = q[seqs].double().cpu().numpy()
    stg = bf16_bits(cache.staging[seqs])
    pool_np = cache.pool.cpu().numpy() if pool_np is None else pool_np
    return oracle.decode_attention(cfg.block_size, cfg.n_q_heads, cfg.n_kv_heads, sign_bits, sm_scale, qn,
                                   pool_np, stg, np.ascontiguousarray(cache.block_table_np[seqs]),
                                   np.asarray(seq_lens, dtype=np.int32)[seqs], flags=int(cfg.flags),
                                   bits=int(cfg.bits))
