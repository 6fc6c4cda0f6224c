"""Seeded synthetic inputs for the five workloads (CPU tensors; no method arithmetic).

This module only draws random numbers and lays them out; it computes nothing
that the library or the oracle computes. Every draw uses a CPU
``torch.Generator`` seeded explicitly; fp32 draws are rounded to bf16 with
round-to-nearest-even where bf16 is asked for, so the GPU and the oracle read
the same bytes.

The shapes and distributions stand in for the pages' workload (a Qwen-sized
75968-column vocabulary shard, 8192 rows) since no dataset or model is used:

1. ``tiny``            N=64, V=4096 fp32, A,B ~ N(0, 2^2); 5% of B set to -inf on 4 rows.
2. ``pages_shape``     N=8192, V=75968 bf16, A,B ~ N(0, 3^2) + per-row offset U[-5, 5].
3. ``numerics_stress`` N=8192, V=75968 fp32 N(0, 3^2) + 1e4 on every row; 1% of B -inf.
4. ``strided``         bf16 [16, 513, 75968] ~ N(0, 3^2), used as x[:, :-1]; and
   ``short_rows``      N=1024 contiguous rows of the ``pages_shape`` distribution.
5. ``linear``          hidden [8192, 4096] ~ N(0, 1), weight [75968, 4096] ~ N(0, 0.02^2), bf16.

Targets are uniform int64 ids in [vocab_start, vocab_start + V); upstream
gradients are N(0, 1) fp32. Sizes may be reduced for parity tests; the recipe
stays the same.
"""
from __future__ import annotations

import torch

VOCAB = 75968
ROWS = 8192


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(gen, shape, sigma):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).mul_(sigma)


def _targets(gen, N, V, vocab_start=0):
    return torch.randint(0, V, (N,), generator=gen, dtype=torch.int64).add_(vocab_start)


def tiny(seed: int = 0, N: int = 64, V: int = 4096, masked_rows: int = 4, mask_frac: float = 0.05):
    gen = _gen(seed)
    a = _normal(gen, (N, V), 2.0)
    b = _normal(gen, (N, V), 2.0)
    rows = torch.randperm(N, generator=gen)[:masked_rows]
    mask = torch.rand(masked_rows, V, generator=gen) < mask_frac
    sub = b[rows]
    sub[mask] = float("-inf")
    b[rows] = sub
    return {"a": a, "b": b, "targets": _targets(gen, N, V), "grad": _normal(gen, (N,), 1.0),
            "masked_rows": rows.sort().values}


def pages_shape(seed: int = 1, N: int = ROWS, V: int = VOCAB, dtype=torch.bfloat16, offset: float = 5.0):
    gen = _gen(seed)
    a = _normal(gen, (N, V), 3.0)
    a += torch.empty(N, 1).uniform_(-offset, offset, generator=gen)
    b = _normal(gen, (N, V), 3.0)
    b += torch.empty(N, 1).uniform_(-offset, offset, generator=gen)
    return {"a": a.to(dtype), "b": b.to(dtype), "targets": _targets(gen, N, V),
            "grad": _normal(gen, (N,), 1.0)}


def numerics_stress(seed: int = 2, N: int = ROWS, V: int = VOCAB, offset: float = 1e4, mask_frac: float = 0.01):
    gen = _gen(seed)
    a = _normal(gen, (N, V), 3.0).add_(offset)
    b = _normal(gen, (N, V), 3.0).add_(offset)
    b[torch.rand(N, V, generator=gen) < mask_frac] = float("-inf")
    return {"a": a, "b": b, "targets": _targets(gen, N, V), "grad": _normal(gen, (N,), 1.0)}


def strided(seed: int = 3, B: int = 16, T: int = 513, V: int = VOCAB, dtype=torch.bfloat16):
    """Full [B, T, V] tensors; the ops read x[:, :-1] in place (B*(T-1) rows)."""
    gen = _gen(seed)
    a = _normal(gen, (B, T, V), 3.0).to(dtype)
    b = _normal(gen, (B, T, V), 3.0).to(dtype)
    return {"a_full": a, "b_full": b, "targets": _targets(gen, B * (T - 1), V).view(B, T - 1),
            "grad": _normal(gen, (B * (T - 1),), 1.0).view(B, T - 1)}


def short_rows(seed: int = 3, N: int = 1024, V: int = VOCAB, dtype=torch.bfloat16):
    return pages_shape(seed=seed + 100, N=N, V=V, dtype=dtype)


def linear(seed: int = 4, N: int = ROWS, V: int = VOCAB, D: int = 4096, dtype=torch.bfloat16):
    gen = _gen(seed)
    h = _normal(gen, (N, D), 1.0).to(dtype)
    w = _normal(gen, (V, D), 0.02).to(dtype)
    return {"hidden": h, "weight": w, "targets": _targets(gen, N, V), "grad": _normal(gen, (N,), 1.0)}


def topk_ids(seed: int, N: int, V: int, K: int, vocab_start: int = 0, ignore_frac: float = 0.1,
             dup_frac: float = 0.1):
    """K target ids per row ([N, K] int64) with upstream gradients [N, K] fp32 ~ N(0, 1).

    Ids are uniform in [vocab_start, vocab_start + V); a share ``dup_frac`` of
    the slots repeats the row's first id (duplicate ids) and a share
    ``ignore_frac`` is -1 (ignored ids).
    """
    gen = _gen(seed)
    t = torch.randint(0, V, (N, K), generator=gen, dtype=torch.int64).add_(vocab_start)
    dup = torch.rand(N, K, generator=gen) < dup_frac
    t = torch.where(dup, t[:, :1].expand(N, K), t)
    t[torch.rand(N, K, generator=gen) < ignore_frac] = -1
    return {"targets": t.contiguous(), "grad": _normal(gen, (N, K), 1.0)}
