"""A multicast between two SM pairs (``cta_pair`` with ``multicast`` 2): a cluster
of four CTAs computes two adjacent 256 x BN tiles of the same rows; each CTA
loads 64 of its half's 128 A rows and multicasts them to the matching CTA of
both pairs, and a ring slot is refilled only after both pairs' MMAs released it.

Parity against the oracle on shapes whose N-tile count leaves the last group's
second tile past N (it loads zeros and stores nothing), ragged M and K, an
M-contiguous A (one 64-element block per CTA), B stored K x N, int8
(bit-exact), the fused bias + activation epilogue, a persistent grid smaller
than the number of tile groups, and the bounded-wait failure path.
"""
import numpy as np
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import oracle
import parity_util as pu

pytestmark = pytest.mark.gpu

# n-blocks of 128 / 256 columns: 1, 3, 5 ... -> groups of two with a partial last group
SHAPES = [(256, 128, 64), (300, 384, 200), (600, 1280, 1000), (1024, 640, 4096)]


def _cfg(bn, **kw):
    return {"block_n": bn, "cta_pair": 1, "multicast": 2, **kw}


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pair_multicast_parity(dtype, bn):
    for M, N, K in SHAPES:
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, _cfg(bn), repeats=2)
        pu.check_full(A, B, dtype, C, "pair mcast bn%d %s %s" % (bn, (M, N, K), dtype))


def test_pair_multicast_int8_bit_exact():
    for M, N, K in ((256, 128, 64), (512, 400, 1040), (1000, 520, 4160)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", _cfg(128))
        pu.check_full(A, B, "i8", C, "i8 pair mcast %s" % ((M, N, K),))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_pair_multicast_layouts(layout):
    for dtype in ("f16", "bf16"):
        for M, N, K in ((256, 264, 192), (600, 520, 1024)):
            A, B = inputs.make_operands(M, N, K, dtype)
            for bn in (128, 256):
                C = pu.run_gpu_layout(A, B, dtype, _cfg(bn), layout)
                pu.check_full(A, B, dtype, C, "%s pair mcast bn%d %s %s" % (layout, bn, (M, N, K), dtype))


def test_pair_multicast_small_persistent_grid_and_epilogue():
    """Two clusters iterate over every tile group; then the fused GELU epilogue."""
    M, N, K = 1024, 2048, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    C = pu.run_gpu(A, B, "f16", _cfg(256, max_ctas=8, raster_group=3), repeats=2)
    pu.check_full(A, B, "f16", C, "pair mcast small grid")
    M, N, K = 512, 1152, 1024
    A, B = inputs.make_operands(M, N, K, "bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(3)).float()
    C = pu.run_gpu_epilogue(A, B, "bf16", _cfg(256), bias, g.ACT_GELU)
    ref = oracle.gemm_tn_half(pu.bits(A), pu.bits(B), oracle.FMT_BF16)
    want = oracle.epilogue(ref, bias.numpy().astype(np.float64), g.ACT_GELU)
    err = np.abs(C.float().cpu().numpy().astype(np.float64) - want)
    tol = 1.13 * pu.tolerance(ref, K) + 1e-2 * np.abs(want) + 1e-6
    assert np.all(err <= tol), float((err - tol).max())


def test_pair_multicast_launch_shape():
    with g.Plan(2048, 2048, 1024, "f16", _cfg(256)) as plan:
        launch = plan.launch
        assert plan.config["multicast"] == 2 and plan.config["cta_pair"] == 1
        assert launch["cluster"] == 4 and launch["grid"] % 4 == 0
        assert launch["max_active_clusters"] == 0 or launch["grid"] <= 4 * launch["max_active_clusters"]


@pytest.mark.parametrize("bn", [128, 256])
def test_pair_multicast_wait_timeout_is_reported(gemm_lib, bn):
    M, N, K = 512, 1024, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", _cfg(bn)) as plan:
        plan.set_timeout(20_000_000)          # 20 ms
        plan.set_wait_test(16)
        plan.run(dA, dB, C)
        with pytest.raises(g.GemmError) as e:
            plan.check()
        assert e.value.status == 9            # GEMM_ERR_DEVICE_TIMEOUT
        plan.set_wait_test(0)
        plan.set_timeout(0)
        plan.run(dA, dB, C)
        plan.check()
    pu.check_full(A, B, "f16", C, "pair mcast bn%d after timeout" % bn)
