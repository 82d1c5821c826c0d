"""GPU tests of gemm_run_splitk_noalloc, the split-K entry point that allocates nothing.

It is for callers that may not allocate device memory (plugins whose host
framework owns all device memory, services with a fixed up-front memory budget,
loops that cannot afford cudaMalloc's synchronisation or failure): its split-K
scratch is a fixed 16 MiB array inside the library.  The tests call it through
the C ABI twice in a row, on different inputs, and compare each result with the
CPU oracle (every element, the parity tolerance) and with the plan entry
point's result (same tile width and split count).  The cases cover a split of
one (no partials), a K that is not a multiple of 64 (a ragged last k-block) and
a split larger than the number of k-blocks (clamped).  This file is collected
last so that a run stopping at the first failure has already run every other
test.
"""
import math

import numpy as np
import pytest
import torch

from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

# (M, N, K, dtype, split_k)
CASES = [
    (200, 136, 2048, "f16", 4),    # four slices of 8 k-blocks, ragged M and N
    (384, 264, 1000, "bf16", 3),   # K % 64 = 40: the last k-block is partly past K
    (136, 200, 520, "f16", 1),     # no split: no partials, plain epilogue
    (72, 64, 136, "bf16", 8),      # 3 k-blocks: the split clamps to 3 slices of one
]


def _tolerance_check(got: torch.Tensor, want: torch.Tensor, K: int):
    g = got.double().cpu().numpy()
    w = want.double().cpu().numpy()
    tol = pu.REL_TOL * np.abs(w) + pu.ABS_TOL_PER_SQRT_K * math.sqrt(K)
    assert np.all(np.abs(g - w) <= tol), float(np.max(np.abs(g - w) - tol))


def test_noalloc_matches_oracle_and_plan_entry_point_two_calls_in_a_row(gemm_lib):
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
        prepared.append((M, N, K, dtype, split, A, B, dA, dB, want, got))
    torch.cuda.synchronize()

    # The first call on this device does the one-time set-up; then every case
    # twice in a row (the second call finds the first one's partials and
    # counters in the shared array).
    M, N, K, dtype, split, A, B, dA, dB, want, got = prepared[0]
    g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, got)
    g.gemm_noalloc_check()
    free_before = torch.cuda.mem_get_info()[0]
    results = []
    for rep in range(2):
        for M, N, K, dtype, split, A, B, dA, dB, want, got in prepared:
            got.fill_(float("nan"))
            torch.cuda.synchronize()
            g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, got)
            g.gemm_noalloc_check()   # synchronises; raises if a wait ran out
            results.append(got.cpu())
    free_after = torch.cuda.mem_get_info()[0]
    # (checked afterwards: the comparisons themselves may make torch's allocator grow)
    for i, (M, N, K, dtype, split, A, B, dA, dB, want, got) in enumerate(prepared * 2):
        where = "noalloc %dx%dx%d %s split %d call %d" % (M, N, K, dtype, split, i // len(CASES))
        pu.check_full(A, B, dtype, results[i], where=where)
        _tolerance_check(results[i], want, K)
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


def test_noalloc_timeout_is_reported_then_the_path_recovers(gemm_lib):
    """A wait that runs out (every ring slot expects 16 bytes that never arrive,
    20 ms limit) is reported by gemm_noalloc_check, which clears it; the next
    normal call is correct and checks clean.  No fault: the kernel's waits are
    bounded and it unwinds on its own."""
    g = gemm_lib
    M, N, K, dtype, split = 200, 136, 2048, "f16", 4
    A, B = inputs.make_operands(M, N, K, dtype)
    dA, dB = A.cuda(), B.cuda()
    C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
    g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, C)   # set-up done before the hook
    g.gemm_noalloc_check()
    try:
        g.gemm_noalloc_set_wait_test(16, 20_000_000)
        g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, C)
        with pytest.raises(g.GemmError) as e:
            g.gemm_noalloc_check()
        assert e.value.status == 9
    finally:
        g.gemm_noalloc_set_wait_test(0, 0)
    g.gemm_noalloc_check()   # the record was cleared by the failed check
    C.fill_(float("nan"))
    g.gemm_run_splitk_noalloc(M, N, K, dtype, split, dA, dB, C)
    g.gemm_noalloc_check()
    pu.check_full(A, B, dtype, C, where="noalloc after a timeout")
