"""The 224-wide SM-pair tile (``cta_pair`` with ``block_n`` 224): a 256 x 224 output
tile per pair, each CTA copying 112 B rows per k-block, a 448-column double
accumulator in a 512-column TMEM allocation, three 64-column TMA stores and the
last 32 columns stored directly from registers.

Parity against the oracle on shapes whose last N tile ends inside each of its
column chunks (a full 64-column store, a store cut by N, the direct 32-column
part cut by N or past it), ragged M and K, two k-blocks per slot, A stored K x M,
the fused bias + activation epilogue, a persistent grid smaller than the tile
count (both accumulator buffers in turn), the bounded-wait failure path, and the
configurations the library refuses.
"""
import numpy as np
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import oracle
import parity_util as pu

pytestmark = pytest.mark.gpu

# N = 224: one tile; 432: the second tile's direct part holds 16 of its 32 columns;
# 1000: the second 64-column store of the last tile is cut by N, the rest is past N;
# 4096: 18 full tiles and one whose first store alone is inside N
SHAPES = [(256, 224, 64), (300, 432, 200), (600, 1000, 1000), (512, 4096, 192), (1024, 672, 4096)]


def _cfg(**kw):
    return {"block_n": 224, "cta_pair": 1, **kw}


@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_bn224_parity(dtype, ks):
    for M, N, K in SHAPES:
        if ks == 2 and K % 64:
            continue
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, _cfg(kblocks_per_stage=ks), repeats=2)
        pu.check_full(A, B, dtype, C, "bn224 ks%d %s %s" % (ks, (M, N, K), dtype))


def test_bn224_a_stored_k_by_m():
    for dtype in ("f16", "bf16"):
        for M, N, K in ((256, 432, 192), (600, 1000, 1024)):
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu_layout(A, B, dtype, _cfg(), "TT")
            pu.check_full(A, B, dtype, C, "TT bn224 %s %s" % ((M, N, K), dtype))


def test_bn224_small_persistent_grid_and_epilogue():
    """Two pairs iterate over every tile; then the fused epilogue on every column chunk."""
    M, N, K = 1024, 2000, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    C = pu.run_gpu(A, B, "f16", _cfg(max_ctas=4, raster_group=3), repeats=2)
    pu.check_full(A, B, "f16", C, "bn224 small grid")
    M, N, K = 512, 1112, 1024
    A, B = inputs.make_operands(M, N, K, "bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(5)).float()
    ref = oracle.gemm_tn_half(pu.bits(A), pu.bits(B), oracle.FMT_BF16)
    for act in (g.ACT_NONE, g.ACT_GELU, g.ACT_SILU):
        C = pu.run_gpu_epilogue(A, B, "bf16", _cfg(), bias, act)
        want = oracle.epilogue(ref, bias.numpy().astype(np.float64), act)
        err = np.abs(C.float().cpu().numpy().astype(np.float64) - want)
        tol = 1.13 * pu.tolerance(ref, K) + 1e-2 * np.abs(want) + 1e-6
        assert np.all(err <= tol), (act, float((err - tol).max()))


def test_bn224_launch_shape():
    with g.Plan(4096, 4096, 1024, "f16", _cfg()) as plan:
        assert plan.config["block_n"] == 224 and plan.config["cta_pair"] == 1
        assert plan.config["stages"] == 6
        launch = plan.launch
        assert launch["cluster"] == 2 and launch["grid"] % 2 == 0
        assert launch["grid"] <= 2 * (16 * 19)          # 16 x 19 tiles of 256 x 224


def test_bn224_refused_configurations():
    for dtype, cfg in (("f16", {"block_n": 224}),                              # one-SM kernel
                       ("i8", {"block_n": 224}),
                       ("f16", _cfg(split_k=2, split_mode=1)),
                       ("f16", _cfg(multicast=2))):
        with pytest.raises(g.GemmError):
            g.Plan(512, 448, 1024, dtype, cfg)
    for layout in ("NN", "NT"):                                                # B stored K x N
        with pytest.raises(g.GemmError):
            g.Plan(512, 448, 1024, "f16", _cfg(), layout=layout)


def test_bn224_wait_timeout_is_reported(gemm_lib):
    M, N, K = 512, 896, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", _cfg()) as plan:
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
    pu.check_full(A, B, "f16", C, "bn224 after timeout")
