"""A-tile multicast: clusters of 2 or 4 CTAs computing adjacent N-tiles of the
same 128 rows, each loading a slice of the shared A tile and multicasting it to
the others (one-SM kernel, ``multicast`` config field).

Parity against the oracle on shapes that span several tile groups, with N-tile
counts that leave the last group partly past N, ragged M and K, every operand
storage the mode supports, int8 (bit-exact), a persistent
grid smaller than the number of groups, and the bounded-wait failure path.
"""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

# (M, N, K): n-blocks of 64 columns = 1, 5, 9, 12 -> groups of 2 or 4 with a
# partial last group; M and K not multiples of the tile.
SHAPES = [(136, 64, 200), (256, 320, 512), (600, 576, 1000), (1024, 768, 4096)]


@pytest.mark.parametrize("mc", [2, 4])
@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_multicast_parity(dtype, bn, mc):
    for M, N, K in SHAPES:
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, {"block_n": bn, "multicast": mc}, repeats=2)
        pu.check_full(A, B, dtype, C, "mcast%d bn%d %s %s" % (mc, bn, (M, N, K), dtype))


@pytest.mark.parametrize("mc", [2, 4])
@pytest.mark.parametrize("bn", [64, 128])
def test_multicast_int8_bit_exact(bn, mc):
    for M, N, K in ((144, 80, 208), (512, 272, 1040), (256, 512, 4096)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", {"block_n": bn, "multicast": mc})
        pu.check_full(A, B, "i8", C, "i8 mcast%d bn%d %s" % (mc, bn, (M, N, K)))


@pytest.mark.parametrize("layout,mc", [("NN", 2), ("NN", 4), ("TT", 2), ("NT", 2)])
def test_multicast_layouts(layout, mc):
    for dtype in ("f16", "bf16"):
        for M, N, K in ((136, 72, 200), (384, 264, 512), (1000, 520, 1024)):
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu_layout(A, B, dtype, {"block_n": 64, "multicast": mc}, layout)
            pu.check_full(A, B, dtype, C, "%s mcast%d %s %s" % (layout, mc, (M, N, K), dtype))


@pytest.mark.parametrize("mc", [2, 4])
def test_multicast_small_persistent_grid(mc):
    """Two clusters iterate over every tile group (grid far below the group count)."""
    M, N, K = 1024, 1024, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    C = pu.run_gpu(A, B, "f16", {"block_n": 64, "multicast": mc, "max_ctas": 2 * mc,
                                 "raster_group": 3})
    pu.check_full(A, B, "f16", C, "mcast%d small grid" % mc)


def test_multicast_config_is_reported():
    with g.Plan(512, 512, 1024, "f16", {"block_n": 64, "multicast": 4}) as plan:
        assert plan.config["multicast"] == 4
    # A stored K x M takes at most two slices; the selected config adapts instead
    with pytest.raises(g.GemmError):
        g.Plan(512, 512, 1024, "f16", {"block_n": 64, "multicast": 4}, layout="TT")


@pytest.mark.parametrize("mc", [2, 4])
def test_multicast_wait_timeout_is_reported(gemm_lib, mc):
    M, N, K = 256, 512, 512
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", {"block_n": 64, "multicast": mc}) as plan:
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
    pu.check_full(A, B, "f16", C, "mcast%d after timeout" % mc)
