"""gemm_run inside a captured CUDA graph (server-mode launch path).

A stream capture records the kernels gemm_run queues (with their tensor maps
and launch attributes); replaying the graph must give the oracle's results,
including after the inputs are refilled in place between replays.
"""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f16", "i8"])
def test_graph_capture_and_replay(gemm_lib, dtype):
    M, N, K = 64, 4096, 64
    A1, B1 = inputs.make_operands(M, N, K, dtype)
    A2, B2 = inputs.make_operands(M, N, K, dtype, seed=99)
    dA, dB = A1.cuda(), B1.cuda()
    C = torch.empty(M, N, dtype=inputs.OUT_DTYPE[dtype], device="cuda")
    stream = torch.cuda.Stream()
    with g.Plan(M, N, K, dtype) as plan:
        plan.run(dA, dB, C, stream)           # first call (tensor maps encoded) outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(8):
                plan.run(dA, dB, C, torch.cuda.current_stream())
        C.zero_()
        graph.replay()
        torch.cuda.synchronize()
        pu.check_full(A1, B1, dtype, C, "graph replay 1")
        dA.copy_(A2.cuda())
        dB.copy_(B2.cuda())
        graph.replay()
        torch.cuda.synchronize()
        plan.check()
        pu.check_full(A2, B2, dtype, C, "graph replay 2")
