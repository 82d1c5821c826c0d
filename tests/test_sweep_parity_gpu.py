"""GPU parity of every benchmarked (shape, configuration) pair against the CPU oracle.

The benchmark's value comes from the 343 fp16 shapes M, N, K in {64, ..., 4096},
each launched with the configuration the library's measured table picks for it
(gemm_plan_create, no explicit configuration), and the named workloads
(8192^3 fp16, the 4096 x 14336 x 4096 bf16 FFN shape, 4096^3 int8 -> int32).
Each is run here exactly that way and compared with the oracle: every element
when M*N*K <= 2^30, else >= 4096 seeded sampled elements (corners and the first
and last row/column of every tile edge included).  The correctness check of the
tuned kernels follows "RL驱动CUDA L2 GEMM内核自动调优：A100/H100 tile size与融合优化"
(correctness paragraph: every tuned kernel is checked against a reference GEMM),
with this library's elementwise tolerance |c - ref| <= 1e-2 |ref| + 1e-3 sqrt(K)
(int8: bit-exact).
"""
import pytest
import torch

from dense_gemm_hgemm_gb300 import inputs, workloads

import parity_util as pu

pytestmark = pytest.mark.gpu

FULL_LIMIT = 1 << 30

SWEEP = workloads.sweep_shapes()
NAMED_EXTRA = [w for w in workloads.NAMED
               if (w.M, w.N, w.K, w.dtype) not in {(s.M, s.N, s.K, s.dtype) for s in SWEEP}]


@pytest.fixture(scope="module")
def sms(gemm_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.cuda.get_device_properties(0).multi_processor_count


def _run_table_config(w, sms):
    import dense_gemm_hgemm_gb300 as g
    A, B = inputs.make_operands(w.M, w.N, w.K, w.dtype, w.a_scale, w.b_scale)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(w.M, w.N, dtype=inputs.OUT_DTYPE[w.dtype], device="cuda")
    with g.Plan(w.M, w.N, w.K, w.dtype) as plan:   # the table's choice, as the benchmark runs it
        want = g.gemm_select_config(w.M, w.N, w.K, w.dtype, sms)
        got = plan.config
        for k in ("block_n", "split_k", "split_mode", "cta_pair", "direct_store", "multicast",
                  "kblocks_per_stage", "raster_group"):
            assert got[k] == want[k], (w.name, k, got, want)
        plan.run(dA, dB, C)
        plan.run(dA, dB, C)    # a second call: split-K counters must have reset themselves
        plan.check()
    return A, B, C


@pytest.mark.parametrize("w", SWEEP, ids=lambda w: "%dx%dx%d" % (w.M, w.N, w.K))
def test_sweep_shape_in_its_tuned_configuration(w, sms):
    A, B, C = _run_table_config(w, sms)
    if w.M * w.N * w.K <= FULL_LIMIT:
        pu.check_full(A, B, w.dtype, C, w.name)
    else:
        pu.check_sampled(A, B, w.dtype, C, count=4096, seed=w.M + w.N + w.K, where=w.name)


@pytest.mark.parametrize("w", NAMED_EXTRA, ids=lambda w: w.name)
def test_named_workload_in_its_tuned_configuration(w, sms):
    A, B, C = _run_table_config(w, sms)
    pu.check_sampled(A, B, w.dtype, C, count=4096, seed=7, where=w.name)
