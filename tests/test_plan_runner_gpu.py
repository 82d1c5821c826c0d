"""Plan.run's per-call form, run(A, B, C, stream) with tensors and a stream, goes
to gemm_run through a C-level runner bound to the plan; every other form takes
the general path.  Both must launch the same kernel: identical results, checked
against the oracle, and the same refusals (a misaligned C, a closed plan)."""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,dtype", [(64, 4096, 64, "f16"), (300, 520, 1040, "bf16"),
                                         (512, 448, 2048, "i8"), (1024, 896, 512, "f16")])
def test_runner_matches_general_path(gemm_lib, M, N, K, dtype):
    A, B = inputs.make_operands(M, N, K, dtype)
    dA, dB = A.cuda(), B.cuda()
    C1 = torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
    C2 = torch.empty_like(C1)
    stream = torch.cuda.Stream()
    with g.Plan(M, N, K, dtype) as plan:
        assert type(plan.run).__name__ == "Runner"
        plan.run(dA, dB, C1, stream)                                  # runner
        g.gemm_run(plan.handle, dA.data_ptr(), dB.data_ptr(), C2.data_ptr(),
                   stream.cuda_stream)                                # general path
        plan.check(stream)
    assert torch.equal(C1.view(torch.int16) if dtype != "i8" else C1,
                       C2.view(torch.int16) if dtype != "i8" else C2)
    pu.check_full(A, B, dtype, C1, "runner %s" % ((M, N, K, dtype),))


def test_runner_refusals(gemm_lib):
    M, N, K = 128, 256, 128
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M * N + 8, dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()
    plan = g.Plan(M, N, K, "f16")
    with pytest.raises(g.GemmError) as e:                 # C at a 2-byte offset
        plan.run(dA, dB, C[1:1 + M * N].view(M, N), stream)
    assert e.value.status == 3                            # GEMM_ERR_ALIGNMENT
    plan.run(dA, dB, C[:M * N].view(M, N), stream)
    plan.check(stream)
    pu.check_full(A, B, "f16", C[:M * N].view(M, N).clone(), "runner after refusal")
    plan.close()
    with pytest.raises(g.GemmError) as e:                 # a closed plan
        plan.run(dA, dB, C[:M * N].view(M, N), stream)
    assert e.value.status == 1                            # GEMM_ERR_INVALID_ARG
