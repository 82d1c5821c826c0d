"""M <= 64 on the one-SM kernel: only the tile's 64 real A rows are copied (a
64-row box, 8 KiB per k-block); the MMA's rows 64..127 read whatever the ring slot
holds and are never stored.  Checked against the oracle in every mode the path
combines with: tile widths 64/128/256, one, two or four k-blocks per slot, both
split-K modes, direct stores, the fused epilogue, M/N-contiguous operands, int8
(bit-exact), and the bounded-wait failure path.  M = 1, 40 and 64 (fewer rows than
the box, and exactly the box).
"""
import numpy as np
import pytest
import torch

import dense_gemm_hgemm_gb300 as g
from dense_gemm_hgemm_gb300 import inputs

import oracle
import parity_util as pu

pytestmark = pytest.mark.gpu

CONFIGS = [
    {"block_n": 64}, {"block_n": 128}, {"block_n": 256},
    {"block_n": 64, "kblocks_per_stage": 2}, {"block_n": 128, "kblocks_per_stage": 2},
    {"block_n": 64, "kblocks_per_stage": 4},
    {"block_n": 64, "split_k": 3}, {"block_n": 64, "split_k": 4, "split_mode": 1},
    {"block_n": 128, "split_k": 8, "split_mode": 1, "kblocks_per_stage": 2},
    {"block_n": 64, "direct_store": 1}, {"block_n": 128, "direct_store": 1, "kblocks_per_stage": 2},
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: "_".join("%s%s" % (k[:2], v) for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 40, 64])
def test_half_a_tile_parity(M, cfg):
    for N, K in ((520, 1024), (4096, 64), (200, 2112)):
        try:       # a cluster split needs equal slices; the library refuses the rest
            g.gemm_workspace_bytes(M, N, K, "f16", cfg)
        except g.GemmError:
            assert cfg.get("split_mode") == 1
            continue
        for dtype in ("f16", "bf16"):
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu(A, B, dtype, cfg, repeats=2)
            pu.check_full(A, B, dtype, C, "half-A M=%d %s %s %s" % (M, cfg, (N, K), dtype))


def test_half_a_tile_int8_bit_exact():
    for M in (16, 64):
        for cfg in ({"block_n": 64}, {"block_n": 128, "kblocks_per_stage": 2},
                    {"block_n": 64, "split_k": 4, "split_mode": 1}, {"block_n": 64, "kblocks_per_stage": 4}):
            A, B = inputs.make_operands(M, 272, 4160, "i8")
            C = pu.run_gpu(A, B, "i8", cfg)
            pu.check_full(A, B, "i8", C, "i8 half-A M=%d %s" % (M, cfg))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_half_a_tile_layouts(layout):
    for M, N, K in ((64, 264, 1088), (40, 520, 256)):
        for dtype in ("f16", "bf16"):
            A, B = inputs.make_operands(M, N, K, dtype)
            for cfg in ({"block_n": 64}, {"block_n": 128, "kblocks_per_stage": 2},
                        {"block_n": 64, "kblocks_per_stage": 4}, {"block_n": 64, "split_k": 3}):
                C = pu.run_gpu_layout(A, B, dtype, cfg, layout)
                pu.check_full(A, B, dtype, C, "%s half-A %s %s %s" % (layout, cfg, (M, N, K), dtype))


def test_half_a_tile_fused_epilogue():
    M, N, K = 64, 1032, 2048
    A, B = inputs.make_operands(M, N, K, "bf16")
    bias = torch.randn(N, generator=torch.Generator().manual_seed(9)).float()
    ref = oracle.gemm_tn_half(pu.bits(A), pu.bits(B), oracle.FMT_BF16)
    for act in (g.ACT_RELU, g.ACT_SILU):
        want = oracle.epilogue(ref, bias.numpy().astype(np.float64), act)
        for cfg in ({"block_n": 64, "kblocks_per_stage": 2}, {"block_n": 64, "split_k": 4, "split_mode": 1}):
            C = pu.run_gpu_epilogue(A, B, "bf16", cfg, bias, act)
            err = np.abs(C.float().cpu().numpy().astype(np.float64) - want)
            tol = 1.13 * pu.tolerance(ref, K) + 1e-2 * np.abs(want) + 1e-6
            assert np.all(err <= tol), (act, cfg, float((err - tol).max()))


def test_half_a_tile_wait_timeout(gemm_lib):
    M, N, K = 64, 1024, 1024
    A, B = inputs.make_operands(M, N, K, "f16")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    with g.Plan(M, N, K, "f16", {"block_n": 64, "kblocks_per_stage": 2}) as plan:
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
    pu.check_full(A, B, "f16", C, "half-A after timeout")
