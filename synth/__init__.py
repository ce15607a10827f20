"""Seeded synthetic inputs for the KVarN KV-cache workloads.

This module holds none of the method's arithmetic: it only draws random
numbers with the shapes and value distributions of the workloads, and the
random sign vector the rotation consumes. Both the CUDA path's tests/bench and
the oracle receive the same tensors from here.

Value model (the pages' workloads are reasoning models whose K/V show a few
outlier channels and widely varying token magnitudes):
    x[t, c] = z[t, c] * m[t] * o[c]
    z ~ N(0, 1);  m[t] = exp(sigma_m * n[t]), n ~ N(0, 1)  (lognormal token scale)
    o[c] = outlier_factor on n_outliers channels picked by a seeded permutation
           per (layer, kv-head), independently for K and V; 1 elsewhere.
Queries are N(0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

_M64 = (1 << 64) - 1


def splitmix64(state: int):
    """One step of SplitMix64 (Steele, Lea, Flood 2014): returns (new_state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & _M64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return state, z ^ (z >> 31)


def sign_bits(seed: int) -> np.ndarray:
    """128 random rotation signs as 4 uint32 words (bit c set => sign -1)."""
    st = seed & _M64
    words = []
    for _ in range(2):
        st, out = splitmix64(st)
        words += [out & 0xFFFFFFFF, out >> 32]
    return np.array(words, dtype=np.uint32)


def outlier_factors(gen: torch.Generator, n_kv: int, n_out: int, factor: float,
                    device) -> torch.Tensor:
    o = torch.ones(n_kv, 128, device=device)
    for h in range(n_kv):
        idx = torch.randperm(128, generator=gen, device=device)[:n_out]
        o[h, idx] = factor
    return o


def kv_values(gen: torch.Generator, batch: int, n_kv: int, L: int, sigma_m: float,
              n_out: int, factor: float, device="cpu") -> torch.Tensor:
    """fp32 [batch][n_kv][L][128] values drawn from the value model."""
    o = outlier_factors(gen, n_kv, n_out, factor, device)
    n = torch.randn(batch, n_kv, L, 1, generator=gen, device=device)
    z = torch.randn(batch, n_kv, L, 128, generator=gen, device=device)
    return z * torch.exp(sigma_m * n) * o[None, :, None, :]


def queries(gen: torch.Generator, batch: int, n_q: int, device="cpu") -> torch.Tensor:
    return torch.randn(batch, n_q, 128, generator=gen, device=device)


def make_gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass
class Workload:
    """Shape and value parameters of one workload."""
    name: str
    n_q: int
    n_kv: int
    block: int
    iters: int
    batch: int
    ctx: int
    sigma_m: float
    n_out: int
    out_factor: float
    dtype: str = "bf16"
    layers: int = 1
    seed: int = 0
    seq_lens: Optional[List[int]] = field(default=None)

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv


# The five workloads (seed = workload index).
TINY = Workload("tiny-1head-256tok", n_q=1, n_kv=1, block=32, iters=3, batch=1, ctx=256,
                sigma_m=1.0, n_out=2, out_factor=10.0, dtype="fp32", seed=0)
LLAMA8B_LAYER = Workload("llama3.1-8b-layer-b16-ctx4096", n_q=32, n_kv=8, block=32, iters=3,
                         batch=16, ctx=4096, sigma_m=1.5, n_out=4, out_factor=20.0, seed=1)
QWEN3_4B_CACHE = Workload("qwen3-4b-36layer-b64-ctx8192", n_q=32, n_kv=8, block=64, iters=2,
                          batch=64, ctx=8192, sigma_m=1.5, n_out=4, out_factor=20.0, layers=36,
                          seed=2)
PHI4_LONG = Workload("phi4-14b-40layer-b8-prefill1k2k-16k-appends", n_q=40, n_kv=10, block=32,
                     iters=3, batch=8, ctx=2048 + 16384, sigma_m=1.5, n_out=4, out_factor=20.0,
                     layers=40, seed=3)


def sweep_point(batch: int, ctx: int, seed: int = 4) -> Workload:
    """Llama-3.1-8B layer shape with ragged lengths ~ U[ctx/2, ctx]."""
    g = np.random.default_rng([seed, batch, ctx])
    lens = g.integers(ctx // 2, ctx + 1, size=batch).tolist()
    return Workload(f"llama3.1-8b-layer-b{batch}-ctx{ctx}-ragged", n_q=32, n_kv=8, block=32,
                    iters=3, batch=batch, ctx=ctx, sigma_m=1.5, n_out=4, out_factor=20.0,
                    seed=seed, seq_lens=lens)


def prefill_lengths(batch: int, lo: int, hi: int, seed: int) -> List[int]:
    g = np.random.default_rng([seed, batch, lo, hi])
    return g.integers(lo, hi + 1, size=batch).tolist()
