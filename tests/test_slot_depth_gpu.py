"""Two 64-wide k-blocks per ring slot (kblocks_per_stage = 2: one-SM kernel,
block_n 64 / 128, each operand's two k-blocks brought by one 3-D copy) against
the oracle (every operand storage): odd k-block counts (the last slot's second k-block is past K and
zero-filled), split-K slices of odd length (the second k-block belongs to the
next slice and is skipped), integer mode (bit-exact), the direct-store and fused
epilogues, the bounded-wait failure path, and the configurations it refuses."""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

KS2 = {"kblocks_per_stage": 2}
# k-blocks of 64: 1, 3, 4, 16, 17 (M and N ragged)
SHAPES = [(128, 64, 64), (136, 72, 192), (256, 320, 256), (600, 576, 1024), (384, 264, 1088)]


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_two_kblock_slots_parity(dtype, bn):
    for M, N, K in SHAPES:
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, {"block_n": bn, **KS2}, repeats=2)
        pu.check_full(A, B, dtype, C, "ks2 bn%d %s %s" % (bn, (M, N, K), dtype))


@pytest.mark.parametrize("split,mode", [(3, 0), (5, 0), (2, 1), (4, 1), (8, 1)])
def test_two_kblock_slots_split_k(split, mode):
    """Slices of odd length end on a slot whose second k-block is the next slice's."""
    for M, N, K in ((128, 128, 1088), (200, 136, 1024), (64, 64, 1536)):
        A, B = inputs.make_operands(M, N, K, "f16")
        for bn in (64, 128):
            cfg = {"block_n": bn, "split_k": split, "split_mode": mode, **KS2}
            try:       # a cluster split needs equal slices; the library refuses the rest
                g.gemm_workspace_bytes(M, N, K, "f16", cfg)
            except g.GemmError:
                assert mode == 1
                continue
            C = pu.run_gpu(A, B, "f16", cfg, repeats=2)
            pu.check_full(A, B, "f16", C, "ks2 split %d/%d bn%d %s" % (split, mode, bn, (M, N, K)))


@pytest.mark.parametrize("bn", [64, 128])
def test_two_kblock_slots_int8_bit_exact(bn):
    for M, N, K in ((144, 80, 192), (512, 272, 1088), (256, 128, 4160)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", {"block_n": bn, **KS2})
        pu.check_full(A, B, "i8", C, "i8 ks2 bn%d %s" % (bn, (M, N, K)))
        C = pu.run_gpu(A, B, "i8", {"block_n": bn, "split_k": 3, **KS2})
        pu.check_full(A, B, "i8", C, "i8 ks2 split3 bn%d %s" % (bn, (M, N, K)))


def test_two_kblock_slots_direct_store():
    for M, N, K in ((130, 72, 192), (257, 520, 1088)):
        for dtype in ("f16", "i8"):
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu(A, B, dtype, {"block_n": 64, "direct_store": 1, **KS2})
            pu.check_full(A, B, dtype, C, "ks2 direct %s %s" % (dtype, (M, N, K)))


def test_two_kblock_slots_refused_where_it_does_not_apply(gemm_lib):
    for shape, layout, bad in (((256, 256, 1024), "TN", {"block_n": 256, **KS2}),
                               ((256, 256, 1024), "TN", {"block_n": 64, "multicast": 2, **KS2}),
                               ((256, 256, 1000), "TN", {"block_n": 64, **KS2}),       # K % 64
                               ((256, 256, 1000), "TT", {"block_n": 64, **KS2}),       # B K-major
                               ((256, 256, 1024), "TN", {"block_n": 64, "kblocks_per_stage": 3}),
                               ((256, 256, 1024), "TN", {"block_n": 64, "stages": 8, **KS2})):
        with pytest.raises(g.GemmError):
            g.Plan(*shape, "f16", bad, layout=layout)
    with g.Plan(256, 256, 1024, "f16", {"block_n": 128, **KS2}) as plan:
        assert plan.config["kblocks_per_stage"] == 2 and plan.config["stages"] == 3


def test_two_kblock_slots_wait_timeout(gemm_lib):
    M, N, K = 256, 320, 1024
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", {"block_n": 64, **KS2}) as plan:
        plan.set_timeout(20_000_000)
        plan.set_wait_test(16)
        plan.run(dA, dB, C)
        with pytest.raises(g.GemmError) as e:
            plan.check()
        assert e.value.status == 9
        plan.set_wait_test(0)
        plan.set_timeout(0)
        plan.run(dA, dB, C)
        plan.check()
    pu.check_full(A, B, "f16", C, "ks2 after timeout")


@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_two_kblock_slots_sm_pair(dtype, bn):
    for M, N, K in ((256, 128, 64), (300, 264, 1088), (1000, 520, 1024)):
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, {"block_n": bn, "cta_pair": 1, **KS2}, repeats=2)
        pu.check_full(A, B, dtype, C, "pair ks2 bn%d %s %s" % (bn, (M, N, K), dtype))
    M, N, K = 512, 384, 1088
    A, B = inputs.make_operands(M, N, K, dtype)
    for s in (2, 4):
        cfg = {"block_n": bn, "cta_pair": 1, "split_k": s, "split_mode": 1, **KS2}
        C = pu.run_gpu(A, B, dtype, cfg)
        pu.check_full(A, B, dtype, C, "pair ks2 split%d bn%d %s" % (s, bn, dtype))


def test_two_kblock_slots_sm_pair_int8():
    for M, N, K in ((256, 128, 1088), (1000, 520, 4160)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", {"block_n": 128, "cta_pair": 1, **KS2})
        pu.check_full(A, B, "i8", C, "i8 pair ks2 %s" % ((M, N, K),))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_two_kblock_slots_layouts(layout):
    """M/N-contiguous operands: two k-blocks per 128-K-row box (K need not be a
    multiple of 64 when both operands are M/N-contiguous)."""
    shapes = [(136, 72, 192), (384, 264, 1088), (1000, 520, 1024)]
    if layout == "NT":
        shapes.append((264, 136, 1000))
    for dtype in ("f16", "bf16"):
        for M, N, K in shapes:
            A, B = inputs.make_operands(M, N, K, dtype)
            for cfg in ({"block_n": 64, **KS2}, {"block_n": 128, **KS2},
                        {"block_n": 256, "cta_pair": 1, **KS2},
                        {"block_n": 64, "split_k": 3, **KS2}):
                C = pu.run_gpu_layout(A, B, dtype, cfg, layout)
                pu.check_full(A, B, dtype, C, "%s ks2 %s %s %s" % (layout, cfg, (M, N, K), dtype))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_two_kblock_slots_layouts_int8(layout):
    for M, N, K in ((144, 80, 192), (512, 272, 1088)):
        A, B = inputs.make_operands(M, N, K, "i8")
        for cfg in ({"block_n": 64, **KS2}, {"block_n": 128, "cta_pair": 1, **KS2}):
            C = pu.run_gpu_layout(A, B, "i8", cfg, layout)
            pu.check_full(A, B, "i8", C, "i8 %s ks2 %s %s" % (layout, cfg, (M, N, K)))
