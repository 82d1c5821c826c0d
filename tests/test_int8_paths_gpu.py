"""int8 -> int32 on the configurations the table uses for large shapes (SM pairs,
128-wide tiles): bit-exact against the oracle, and against the other int8 paths.

Covers ragged M, N and K (K below one k-block, odd k-block counts, K just past a
1024-wide exact-accumulation chunk), the largest magnitudes (every product 2^14,
sums past 2^24 that only the int32 chunk sums keep exact), int32 wrap-around,
persistent pairs that walk several tiles, agreement of the SM-pair, SM-pair
split-K and one-SM kernels, and the bounded-wait failure path.
"""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

PAIR = {"block_n": 128, "cta_pair": 1}

# (M, N, K): K in 16-byte multiples; 16 (< one k-block), 80 (two k-blocks, the
# second partial), 208, 1040 (one full chunk + one k-block), 2064, 4112.
SHAPES = [(256, 128, 16), (300, 136, 80), (520, 264, 208), (256, 384, 1040), (200, 72, 2064),
          (513, 260, 4112)]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_pair_bit_exact(shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "i8")
    C = pu.run_gpu(A, B, "i8", PAIR, repeats=2)
    pu.check_full(A, B, "i8", C, "i8 pair %s" % (shape,))


def test_pair_extremes():
    """(-128)(-128) * K: every fp32 chunk sum is 2^24 exactly; the total 2^26 needs
    the int32 chunk sums."""
    K = 4096
    for a, b in ((-128, -128), (-128, 127), (127, 127)):
        A = torch.full((384, K), a, dtype=torch.int8)
        B = torch.full((256, K), b, dtype=torch.int8)
        C = pu.run_gpu(A, B, "i8", PAIR)
        assert torch.all(C.cpu() == a * b * K), (a, b)


def test_pair_wraps_mod_2_32():
    """Sums past 2^31 wrap like int32 arithmetic (the oracle's definition)."""
    K = 4096 * 33          # 33 x 4096 x 2^14 > 2^31
    A = torch.full((256, K), -128, dtype=torch.int8)
    B = torch.full((128, K), -128, dtype=torch.int8)
    C = pu.run_gpu(A, B, "i8", PAIR)
    want = (128 * 128 * K) & 0xFFFFFFFF
    want = want - (1 << 32) if want >= (1 << 31) else want
    assert torch.all(C.cpu() == want)


@pytest.mark.parametrize("raster", [1, 3])
def test_pair_persistent(raster):
    """Two SM pairs walk all 24 tiles (several units per pair)."""
    M, N, K = 1024, 768, 1104
    A, B = inputs.make_operands(M, N, K, "i8")
    C = pu.run_gpu(A, B, "i8", {**PAIR, "max_ctas": 4, "raster_group": raster})
    pu.check_full(A, B, "i8", C, "i8 pair, 2 pairs, raster %d" % raster)


def test_int8_paths_agree():
    """Same int32 result from the SM-pair kernel, the SM-pair split-K kernel and the
    one-SM kernel."""
    M, N, K = 640, 392, 2048
    A, B = inputs.make_operands(M, N, K, "i8")
    c0 = pu.run_gpu(A, B, "i8", PAIR)
    c1 = pu.run_gpu(A, B, "i8", {"block_n": 128, "cta_pair": 1, "split_k": 2, "split_mode": 1})
    c2 = pu.run_gpu(A, B, "i8", {"block_n": 128})
    assert torch.equal(c0, c1) and torch.equal(c0, c2)
    pu.check_full(A, B, "i8", c0, "i8 paths")


def test_pair_wait_timeout_is_reported(gemm_lib):
    M, N, K = 512, 256, 2048
    A, B = inputs.make_operands(M, N, K, "i8")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.int32, device="cuda")
    with g.Plan(M, N, K, "i8", PAIR) as plan:
        plan.set_timeout(20_000_000)          # 20 ms
        plan.set_wait_test(16)                # a ring slot never completes
        plan.run(dA, dB, C)
        with pytest.raises(g.GemmError) as e:
            plan.check()
        assert e.value.status == 9            # GEMM_ERR_DEVICE_TIMEOUT
        plan.set_wait_test(0)
        plan.set_timeout(0)
        plan.run(dA, dB, C)
        plan.check()
    pu.check_full(A, B, "i8", C, "i8 pair after timeout")
