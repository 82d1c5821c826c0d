"""Helpers shared by the GPU parity tests: run the CUDA path, ask the oracle, compare.

Comparison rule for fp16/bf16 (elementwise, on every checked element):
    |C_gpu - ref| <= 1e-2 * |ref| + 1e-3 * sqrt(K)
where ref is the oracle's fp64 sum of the exactly decoded inputs.  int8 -> int32
results must equal the oracle's wrapped int32 bit for bit.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from dense_gemm_hgemm_gb300 import inputs

REL_TOL = 1e-2
ABS_TOL_PER_SQRT_K = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def fmt(dtype: str) -> int:
    return oracle.FMT_F16 if dtype in ("f16", "i8") else oracle.FMT_BF16


def run_gpu(A: torch.Tensor, B: torch.Tensor, dtype: str, config=None, out=None,
            repeats: int = 1) -> torch.Tensor:
    """C = A @ B.T through the C ABI; A, B CPU or CUDA tensors."""
    import dense_gemm_hgemm_gb300 as g
    M, K = A.shape
    N = B.shape[0]
    dA = A.cuda() if not A.is_cuda else A
    dB = B.cuda() if not B.is_cuda else B
    C = out if out is not None else torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
    with g.Plan(M, N, K, dtype, config) as plan:
        for _ in range(repeats):
            plan.run(dA, dB, C)
        plan.check()
    return C


def tolerance(ref: np.ndarray, K: int) -> np.ndarray:
    return REL_TOL * np.abs(ref) + ABS_TOL_PER_SQRT_K * math.sqrt(max(K, 1))


def assert_close_half(C: np.ndarray, ref: np.ndarray, K: int, where: str = ""):
    err = np.abs(C.astype(np.float64) - ref)
    tol = tolerance(ref, K)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError("%s: %d/%d elements out of tolerance; first at %s: gpu=%r ref=%r "
                             "tol=%r" % (where, bad.sum(), bad.size, i, C[i], ref[i], tol[i]))
    # secondary, reported: Frobenius-norm relative error
    denom = np.linalg.norm(ref)
    return float(np.linalg.norm(C.astype(np.float64) - ref) / denom) if denom > 0 else 0.0


def check_full(A: torch.Tensor, B: torch.Tensor, dtype: str, C_gpu: torch.Tensor, where=""):
    K = A.shape[1]
    if dtype == "i8":
        _, c32 = oracle.gemm_tn_i8(A.numpy(), B.numpy())
        got = C_gpu.cpu().numpy()
        if not np.array_equal(got, c32):
            bad = np.argwhere(got != c32)
            i = tuple(bad[0])
            raise AssertionError("%s: %d int32 mismatches; first at %s: gpu=%d ref=%d"
                                 % (where, len(bad), i, got[i], c32[i]))
        return 0.0
    ref = oracle.gemm_tn_half(bits(A), bits(B), fmt(dtype))
    return assert_close_half(C_gpu.float().cpu().numpy(), ref, K, where)


def check_sampled(A: torch.Tensor, B: torch.Tensor, dtype: str, C_gpu: torch.Tensor,
                  count: int = 4096, seed: int = 1234, where=""):
    M, K = A.shape
    N = B.shape[0]
    rows, cols = inputs.sample_positions(M, N, count, seed)
    got = C_gpu[rows.cuda(), cols.cuda()].cpu()
    if dtype == "i8":
        _, o32 = oracle.gemm_tn_i8_sampled(A.numpy(), B.numpy(), rows.numpy(), cols.numpy())
        g = got.numpy()
        if not np.array_equal(g, o32):
            bad = np.flatnonzero(g != o32)
            raise AssertionError("%s: %d sampled int32 mismatches; first (%d,%d) gpu=%d ref=%d"
                                 % (where, len(bad), rows[bad[0]], cols[bad[0]], g[bad[0]],
                                    o32[bad[0]]))
        return 0.0
    ref = oracle.gemm_tn_half_sampled(bits(A), bits(B), fmt(dtype), rows.numpy(), cols.numpy())
    return assert_close_half(got.float().numpy(), ref, K, where)


def run_gpu_epilogue(A, B, dtype, config, bias, act):
    """C = act(A @ B.T + bias) through gemm_run_bias_act."""
    import dense_gemm_hgemm_gb300 as g
    M, K = A.shape
    N = B.shape[0]
    C = torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
    db = None if bias is None else bias.cuda()
    with g.Plan(M, N, K, dtype, config) as plan:
        plan.run(A.cuda(), B.cuda(), C, bias=db, act=act)
        plan.check()
    return C


def stored(A: torch.Tensor, B: torch.Tensor, layout: str):
    """A[M,K], B[N,K] (the logical TN operands) in the storage of `layout`."""
    a = A.T.contiguous() if layout in ("TT", "NT") else A
    b = B.T.contiguous() if layout in ("NN", "NT") else B
    return a, b


def run_gpu_layout(A, B, dtype, config, layout):
    """C = A @ B.T computed from A, B stored as `layout` prescribes."""
    import dense_gemm_hgemm_gb300 as g
    M, K = A.shape
    N = B.shape[0]
    a, b = stored(A, B, layout)
    C = torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
    with g.Plan(M, N, K, dtype, config, layout=layout) as plan:
        plan.run(a.cuda(), b.cuda(), C)
        plan.run(a.cuda(), b.cuda(), C)
        plan.check()
    return C
