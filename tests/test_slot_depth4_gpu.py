"""Four 64-wide k-blocks per ring slot (kblocks_per_stage = 4: one-SM kernel with
block_n 64 and SM-pair kernel with block_n 128, two 96 KiB slots, each operand's
four k-blocks brought by one 3-D copy) against the oracle: k-block counts that
are not multiples of four (the last slot's later k-blocks lie past K and are
zero-filled), split-K slices whose length is not a multiple of four (a slot's
later k-blocks belong to the next slice and are skipped), integer mode
(bit-exact), direct stores, the fused epilogue, every operand storage, the
bounded-wait failure path, and the configurations it refuses."""
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

KS4 = {"kblocks_per_stage": 4}
ONE_SM = {"block_n": 64, **KS4}
PAIR = {"block_n": 128, "cta_pair": 1, **KS4}
# k-blocks of 64: 1, 3, 4, 5, 17 (M and N ragged)
SHAPES = [(128, 64, 64), (136, 72, 192), (256, 320, 256), (600, 576, 320), (384, 264, 1088)]


@pytest.mark.parametrize("cfg", [ONE_SM, PAIR], ids=["one_sm_bn64", "pair_bn128"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_four_kblock_slots_parity(dtype, cfg):
    for M, N, K in SHAPES:
        A, B = inputs.make_operands(M, N, K, dtype)
        C = pu.run_gpu(A, B, dtype, cfg, repeats=2)
        pu.check_full(A, B, dtype, C, "ks4 %s %s %s" % (cfg, (M, N, K), dtype))


@pytest.mark.parametrize("split,mode", [(3, 0), (5, 0), (2, 1), (4, 1), (8, 1)])
def test_four_kblock_slots_split_k(split, mode):
    """Slices of 5, 6, 7 or 9 k-blocks end inside a slot."""
    for M, N, K in ((128, 128, 1088), (200, 136, 1024), (64, 64, 1536), (512, 384, 1216)):
        A, B = inputs.make_operands(M, N, K, "f16")
        for base in (ONE_SM, PAIR):
            cfg = {**base, "split_k": split, "split_mode": mode}
            try:       # a cluster split needs equal slices; pairs split only in the cluster
                g.gemm_workspace_bytes(M, N, K, "f16", cfg)
            except g.GemmError:
                continue
            C = pu.run_gpu(A, B, "f16", cfg, repeats=2)
            pu.check_full(A, B, "f16", C, "ks4 split %d/%d %s %s" % (split, mode, base, (M, N, K)))


@pytest.mark.parametrize("cfg", [ONE_SM, PAIR], ids=["one_sm_bn64", "pair_bn128"])
def test_four_kblock_slots_int8_bit_exact(cfg):
    """Integer mode restarts the exact fp32 accumulation every 16 k-blocks (four slots)."""
    for M, N, K in ((144, 80, 192), (512, 272, 1088), (256, 128, 4160)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu(A, B, "i8", cfg)
        pu.check_full(A, B, "i8", C, "i8 ks4 %s %s" % (cfg, (M, N, K)))
    A = torch.full((256, 4096), -128, dtype=torch.int8)
    B = torch.full((128, 4096), -128, dtype=torch.int8)
    B[1::2] = 127
    C = pu.run_gpu(A, B, "i8", cfg).cpu()
    assert torch.all(C[:, 0::2] == 4096 * 16384) and torch.all(C[:, 1::2] == -128 * 127 * 4096)


def test_four_kblock_slots_direct_store_and_epilogue():
    for M, N, K in ((130, 72, 192), (257, 520, 1088)):
        for dtype in ("f16", "i8"):
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu(A, B, dtype, {**ONE_SM, "direct_store": 1})
            pu.check_full(A, B, dtype, C, "ks4 direct %s %s" % (dtype, (M, N, K)))
    import numpy as np
    import oracle
    M, N, K = 300, 264, 1088
    A, B = inputs.make_operands(M, N, K, "bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(5)).float()
    for cfg in (ONE_SM, PAIR):
        C = pu.run_gpu_epilogue(A, B, "bf16", cfg, bias, g.ACT_GELU)
        ref = oracle.gemm_tn_half(pu.bits(A), pu.bits(B), oracle.FMT_BF16)
        want = oracle.epilogue(ref, bias.numpy().astype(np.float64), g.ACT_GELU)
        err = np.abs(C.float().cpu().numpy().astype(np.float64) - want)
        # the GEMM rule scaled by GELU's Lipschitz bound, plus the output rounding
        tol = 1.13 * pu.tolerance(ref, K) + 1e-2 * np.abs(want) + 1e-6
        assert np.all(err <= tol), ("ks4 gelu", cfg, float((err - tol).max()))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_four_kblock_slots_layouts(layout):
    """M/N-contiguous operands: four k-blocks per 256-K-row box."""
    for dtype in ("f16", "bf16"):
        for M, N, K in ((136, 72, 192), (384, 264, 1088), (1000, 520, 1024)):
            A, B = inputs.make_operands(M, N, K, dtype)
            for cfg in (ONE_SM, PAIR, {**ONE_SM, "split_k": 3}):
                C = pu.run_gpu_layout(A, B, dtype, cfg, layout)
                pu.check_full(A, B, dtype, C, "%s ks4 %s %s %s" % (layout, cfg, (M, N, K), dtype))
    M, N, K = 512, 272, 1088
    A, B = inputs.make_operands(M, N, K, "i8")
    for cfg in (ONE_SM, PAIR):
        C = pu.run_gpu_layout(A, B, "i8", cfg, layout)
        pu.check_full(A, B, "i8", C, "i8 %s ks4 %s" % (layout, cfg))


def test_four_kblock_slots_refused_where_it_does_not_apply(gemm_lib):
    for shape, layout, bad in (((256, 256, 1024), "TN", {"block_n": 128, **KS4}),
                               ((256, 256, 1024), "TN", {"block_n": 256, "cta_pair": 1, **KS4}),
                               ((256, 256, 1000), "TN", ONE_SM),                      # K % 64
                               ((256, 256, 1024), "TN", {**ONE_SM, "stages": 4})):
        with pytest.raises(g.GemmError):
            g.Plan(*shape, "f16", bad, layout=layout)
    with g.Plan(256, 256, 1024, "f16", PAIR) as plan:
        assert plan.config["kblocks_per_stage"] == 4 and plan.config["stages"] == 2


@pytest.mark.parametrize("cfg", [ONE_SM, PAIR], ids=["one_sm_bn64", "pair_bn128"])
def test_four_kblock_slots_wait_timeout(gemm_lib, cfg):
    M, N, K = 256, 320, 1024
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", cfg) as plan:
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
    pu.check_full(A, B, "f16", C, "ks4 after timeout")
