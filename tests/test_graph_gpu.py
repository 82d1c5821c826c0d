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


def test_vectorcall_and_ctypes_paths_agree(gemm_lib, monkeypatch):
    """Plan.run through the vectorcall entry point and through ctypes (the path used
    when the module cannot be built) launch the same kernel: identical bytes, for
    every way of passing the stream."""
    M, N, K = 192, 320, 384
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    s = torch.cuda.Stream()
    outs = []
    for fast in (True, False):
        if not fast:
            monkeypatch.setattr(g, "_pycall", None)
        with g.Plan(M, N, K, "f16") as plan:
            for stream in (s, s.cuda_stream, None):
                C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
                with torch.cuda.stream(s):
                    plan.run(dA, dB, C, stream)
                plan.check(s)
                torch.cuda.synchronize()
                outs.append(C)
            # raw device addresses as ints
            C = torch.zeros(M, N, dtype=torch.float16, device="cuda")
            plan.run(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), s)
            plan.check(s)
            outs.append(C)
    for C in outs[1:]:
        assert torch.equal(C.view(torch.int16), outs[0].view(torch.int16))
    pu.check_full(A, B, "f16", outs[0], "vectorcall vs ctypes")
