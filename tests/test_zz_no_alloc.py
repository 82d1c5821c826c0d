"""GPU test of gemm_run_splitk_noalloc, the split-K entry point that allocates nothing.

It is for callers that may not allocate device memory (plugins whose host
framework owns all device memory, services with a fixed up-front memory budget,
loops that cannot afford cudaMalloc's synchronisation or failure): its split-K
scratch is a fixed 16 MiB array inside the library.  The test calls it through
the C ABI twice in a row, on different inputs, and compares each result with the
plan entry point's (same tile width and split count) under the parity
tolerance.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

CASES = [(200, 136, 2048, "f16", 4), (384, 264, 1000, "bf16", 3)]


def _tolerance_check(got: torch.Tensor, want: torch.Tensor, K: int):
    g = got.double().cpu().numpy()
    w = want.double().cpu().numpy()
    tol = pu.REL_TOL * np.abs(w) + pu.ABS_TOL_PER_SQRT_K * math.sqrt(K)
    assert np.all(np.abs(g - w) <= tol), float(np.max(np.abs(g - w) - tol))


def test_noalloc_matches_plan_entry_point_two_calls_in_a_row(gemm_lib):
    g = gemm_lib
    assert torch.cuda.is_available()
    prepared = []
    for M, N, K, dtype, split in CASES:
        A, B = inputs.make_operands(M, N, K, dtype)
        dA, dB = A.cuda(), B.cuda()
        want = torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
        with g.Plan(M, N, K, dtype, {"block_n": 64, "split_k": split}) as plan:
            plan.run(dA, dB, want)
            plan.check()
        got = torch.full((M, N), float("nan"), dtype=inputs.OUT_DTYPE[dtype], device="cuda")
        prepared.append((M, N, K, dtype, split, dA, dB, want, got))
    torch.cuda.synchronize()

    # First call on this device does the one-time set-up; then two calls in a row.
    M, N, K, dtype, split, dA, dB, want, got = prepared[0]
    g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, got)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for M, N, K, dtype, split, dA, dB, want, got in prepared:
        got.fill_(float("nan"))
        torch.cuda.synchronize()
        g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, got)
        torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    # (checked afterwards: the comparison itself may make torch's allocator grow)
    for M, N, K, dtype, split, dA, dB, want, got in prepared:
        _tolerance_check(got, want, K)
    assert free_after == free_before   # the calls allocated nothing


def test_noalloc_rejects_problems_beyond_its_scratch(gemm_lib):
    g = gemm_lib
    A = torch.zeros(4096, 1024, dtype=torch.float16, device="cuda")
    B = torch.zeros(4096, 1024, dtype=torch.float16, device="cuda")
    C = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_run_splitk_noalloc(4096, 4096, 1024, "f16", 2, A, B, C)   # 2048 tiles x 2 slices
    assert e.value.status == 11
    with pytest.raises(g.GemmError) as e:
        g.gemm_run_splitk_noalloc(64, 64, 64, "i8", 1, A, B, C)
    assert e.value.status == 2
