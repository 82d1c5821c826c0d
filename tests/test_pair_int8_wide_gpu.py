"""int8 -> int32 on 224- and 256-wide SM-pair tiles.  Each 1024-long K chunk is an
exact fp32 sum in TMEM; eight epilogue warps (two per TMEM lane quarter: columns
[0, 128) and [128, BN) of the same 32 rows) round every chunk to int32 and add it
to their register sums (mod 2^32), which are stored once per tile.

Bit-exact against the oracle for one to five chunks per tile, ragged M and N
(boxes cut by N), two k-blocks per slot, persistent pairs that run several tiles,
A and B stored K-major or not; plus closed-form cases: the largest products, a
chunk sum of 2^24 - 2^14 + 1, and a sum past 2^31 that must wrap like int32.
"""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

# K = 64: one chunk (stores only); 1040: 16 + 1 k-blocks; 4160: five chunks
SHAPES = [(256, 224, 64), (300, 264, 1040), (1000, 520, 4160), (512, 2048, 2048)]


def _cfg(bn, **kw):
    return {"block_n": bn, "cta_pair": 1, **kw}


@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("bn", [224, 256])
def test_wide_int8_bit_exact(bn, ks):
    for M, N, K in SHAPES:
        if ks == 2 and K % 64:
            continue
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", _cfg(bn, kblocks_per_stage=ks), repeats=2)
        pu.check_full(A, B, "i8", C, "i8 bn%d ks%d %s" % (bn, ks, (M, N, K)))


@pytest.mark.parametrize("bn", [224, 256])
def test_wide_int8_persistent_pairs(bn):
    """Two pairs run every tile in turn: chunk counts restart per tile."""
    M, N, K = 1024, 1000, 2112
    A, B = inputs.make_operands(M, N, K, "i8")
    C = pu.run_gpu(A, B, "i8", _cfg(bn, max_ctas=4, raster_group=3), repeats=2)
    pu.check_full(A, B, "i8", C, "i8 bn%d small grid" % bn)


@pytest.mark.parametrize("layout", ["TT", "NN", "NT"])
def test_wide_int8_layouts(layout):
    M, N, K = 512, 448, 2048
    A, B = inputs.make_operands(M, N, K, "i8")
    for bn in (224, 256):
        if bn == 224 and layout in ("NN", "NT"):     # B stored K x N: 256 only
            continue
        C = pu.run_gpu_layout(A, B, "i8", _cfg(bn), layout)
        pu.check_full(A, B, "i8", C, "i8 %s bn%d" % (layout, bn))


@pytest.mark.parametrize("bn", [224, 256])
def test_wide_int8_extremes(bn):
    K = 4096
    A = torch.full((384, K), -128, dtype=torch.int8)
    B = torch.full((448, K), -128, dtype=torch.int8)
    B[1::2] = 127
    C = pu.run_gpu(A, B, "i8", _cfg(bn)).cpu()
    assert torch.all(C[:, 0::2] == K * 16384)
    assert torch.all(C[:, 1::2] == -128 * 127 * K)


@pytest.mark.parametrize("bn", [224, 256])
def test_wide_int8_small_addend_at_top_of_range(bn):
    """Per chunk 1023 products of 2^14 and one of 1: 2^24 - 2^14 + 1 per chunk."""
    K = 4096
    A = torch.full((256, K), -128, dtype=torch.int8)
    B = torch.full((256, K), -128, dtype=torch.int8)
    for c in range(K // 1024):
        A[:, c * 1024 + 1023] = 1
        B[:, c * 1024 + 1023] = 1
    A[1::2, ::2] = 127
    C = pu.run_gpu(A, B, "i8", _cfg(bn)).cpu()
    assert torch.all(C[0::2] == 4 * (1023 * 16384 + 1))
    pu.check_full(A, B, "i8", C, "i8 small addend bn%d" % bn)


@pytest.mark.parametrize("bn", [224, 256])
def test_wide_int8_wraps_like_int32(bn):
    """132 chunks of 2^24 each: 2214592512 > 2^31 - 1 wraps to -2080374784."""
    K = 132 * 1024
    A = torch.full((256, K), -128, dtype=torch.int8)
    B = torch.full((224, K), -128, dtype=torch.int8)
    C = pu.run_gpu(A, B, "i8", _cfg(bn)).cpu()
    want = (K * 16384 + 2**31) % 2**32 - 2**31
    assert want == -2080374784
    assert torch.all(C == want)


def test_wide_int8_wait_timeout_is_reported(gemm_lib):
    M, N, K = 512, 512, 2048
    A, B = inputs.make_operands(M, N, K, "i8")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.int32, device="cuda")
    with g.Plan(M, N, K, "i8", _cfg(256)) as plan:
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
    pu.check_full(A, B, "i8", C, "i8 bn256 after timeout")
