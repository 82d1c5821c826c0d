"""Seeded synthetic operands for the TN GEMM.

This module is the one piece shared by the CUDA path's callers and the CPU
oracle's callers: it only draws random numbers (torch's CPU generator, so the
same seed gives the same bits on x86-64 and aarch64) and holds none of the
GEMM's arithmetic.  It imports nothing from the rest of the package.

Recipe (per shape):
  * seed  = (M*1000003 + N*1009 + K)*4 + dtype_id   (f16=0, bf16=1, i8=2)
  * A is drawn from a generator seeded with ``seed``, B from ``seed ^ 0x5bd1e995``.
  * fp16/bf16: float32 N(0,1) samples times a per-operand scale, rounded to the
    operand type (round-to-nearest-even).
  * int8: uniform integers in [-128, 127], both ends included.
"""
from __future__ import annotations

import torch

DTYPE_ID = {"f16": 0, "bf16": 1, "i8": 2}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int8}
OUT_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "i8": torch.int32}


def shape_seed(M: int, N: int, K: int, dtype: str) -> int:
    return ((M * 1000003 + N * 1009 + K) * 4 + DTYPE_ID[dtype]) & 0x7FFFFFFFFFFFFFFF


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _normal(rows: int, cols: int, scale: float, dtype: str, seed: int) -> torch.Tensor:
    x = torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(TORCH_DTYPE[dtype])


def _uniform_i8(rows: int, cols: int, seed: int) -> torch.Tensor:
    return torch.randint(-128, 128, (rows, cols), generator=_gen(seed), dtype=torch.int8)


def make_operands(M: int, N: int, K: int, dtype: str, a_scale: float = 1.0,
                  b_scale: float = 1.0, seed: int | None = None):
    """Return CPU tensors A[M,K], B[N,K] (row-major, K contiguous) for one shape."""
    if seed is None:
        seed = shape_seed(M, N, K, dtype)
    seed_b = seed ^ 0x5BD1E995
    if dtype == "i8":
        return _uniform_i8(M, K, seed), _uniform_i8(N, K, seed_b)
    return (_normal(M, K, a_scale, dtype, seed), _normal(N, K, b_scale, dtype, seed_b))


def small_integers(rows: int, cols: int, lo: int, hi: int, dtype: str, seed: int) -> torch.Tensor:
    """Integers drawn uniformly from [lo, hi], stored in ``dtype`` (exact there)."""
    x = torch.randint(lo, hi + 1, (rows, cols), generator=_gen(seed), dtype=torch.int32)
    return x.to(TORCH_DTYPE[dtype])


def constant(rows: int, cols: int, value: float, dtype: str) -> torch.Tensor:
    return torch.full((rows, cols), value, dtype=TORCH_DTYPE[dtype])


def sample_positions(M: int, N: int, count: int, seed: int, tile_m: int = 128,
                     tile_n: int = 64):
    """Seeded output positions for sampled checks of large results.

    Holds the four corners, the first and last row/column of every tile edge
    class along each axis (for the given tile sizes), and ``count`` positions
    drawn without replacement by a seeded generator.
    """
    g = _gen(seed)
    total = M * N
    count = min(count, total)
    lin = torch.randperm(total, generator=g)[:count] if total <= (1 << 26) else \
        torch.randint(0, total, (count,), generator=g)
    rows = (lin // N).tolist()
    cols = (lin % N).tolist()
    extra = set()
    for r in (0, M - 1):
        for c in (0, N - 1):
            extra.add((r, c))
    edge_rows = sorted({min(M - 1, x) for t in range(0, M, tile_m) for x in (t, t + tile_m - 1)})
    edge_cols = sorted({min(N - 1, x) for t in range(0, N, tile_n) for x in (t, t + tile_n - 1)})
    for i, r in enumerate(edge_rows[:64]):
        extra.add((r, edge_cols[i % len(edge_cols)]))
    for i, c in enumerate(edge_cols[:64]):
        extra.add((edge_rows[i % len(edge_rows)], c))
    have = set(zip(rows, cols))
    for rc in sorted(extra):
        if rc not in have:
            rows.append(rc[0])
            cols.append(rc[1])
    return torch.tensor(rows, dtype=torch.int64), torch.tensor(cols, dtype=torch.int64)
