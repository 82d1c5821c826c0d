"""Fused linear-layer epilogue C = act(A @ B.T + bias) against the oracle.

Tolerance: the GEMM rule propagated through the activation (Lipschitz constant
<= 1.13 for GELU, 1.1 for SiLU, 1 for ReLU) plus the output rounding:
    |c - act(ref + b)| <= 1.13 * (1e-2 * |ref| + 1e-3 * sqrt(K)) + 1e-2 * |act(ref + b)| + 1e-6
"""
import math

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_hgemm_gb300 import inputs, workloads

import parity_util as pu

pytestmark = pytest.mark.gpu

MODES = [
    ("one_sm_tma", (300, 264, 1000), {"block_n": 128}),
    ("one_sm_direct", (130, 72, 208), {"block_n": 64, "direct_store": 1}),
    ("workspace_split", (200, 136, 1024), {"block_n": 64, "split_k": 3}),
    ("cluster_split", (128, 256, 2048), {"block_n": 64, "split_k": 4, "split_mode": 1}),
    ("cluster_split2", (260, 200, 1536), {"block_n": 128, "split_k": 2, "split_mode": 1}),
    ("cluster_split8", (136, 520, 2048), {"block_n": 256, "split_k": 8, "split_mode": 1}),
    ("sm_pair", (1000, 520, 512), {"block_n": 256, "cta_pair": 1}),
    ("multicast2", (300, 264, 1000), {"block_n": 64, "multicast": 2}),
    ("multicast4", (200, 520, 640), {"block_n": 128, "multicast": 4}),
    ("pair_split", (300, 264, 1024), {"block_n": 256, "cta_pair": 1, "split_k": 4,
                                      "split_mode": 1}),
    ("pair_split2", (520, 136, 1024), {"block_n": 128, "cta_pair": 1, "split_k": 2,
                                       "split_mode": 1}),
    ("two_kblock_slots", (300, 264, 1088), {"block_n": 128, "kblocks_per_stage": 2}),
    # plain plans launch the epilogue form for a fused call: 256-wide one-SM tiles,
    # SM pairs of 128- and 224-wide tiles (the last 32 columns stored per thread),
    # ragged N
    ("one_sm_256", (260, 600, 512), {"block_n": 256}),
    ("sm_pair_128", (520, 200, 640), {"block_n": 128, "cta_pair": 1}),
    ("sm_pair_224", (600, 472, 512), {"block_n": 224, "cta_pair": 1}),
    ("half_a", (64, 520, 512), {"block_n": 128}),   # M <= 64: the 64-row A box
]


def _check(A, B, dtype, C, bias, act, where, rows=None, cols=None):
    K = A.shape[1]
    fmt = pu.fmt(dtype)
    if rows is None:
        pre = oracle.gemm_tn_half(pu.bits(A), pu.bits(B), fmt)
        want = oracle.epilogue(pre, bias, act)
        got = C.float().cpu().numpy().astype(np.float64)
    else:
        pre = oracle.gemm_tn_half_sampled(pu.bits(A), pu.bits(B), fmt, rows, cols)
        want = oracle.epilogue_sampled(pre, cols, bias, act)
        got = C[torch.as_tensor(rows).cuda(), torch.as_tensor(cols).cuda()].float().cpu().numpy()
    tol = 1.13 * (1e-2 * np.abs(pre) + 1e-3 * math.sqrt(K)) + 1e-2 * np.abs(want) + 1e-6
    bad = ~(np.abs(got - want) <= tol)
    assert not bad.any(), "%s: %d bad, first gpu=%r want=%r" % (where, bad.sum(), got[bad][0], want[bad][0])


@pytest.mark.parametrize("act", [0, 1, 2, 3], ids=["none", "relu", "gelu", "silu"])
@pytest.mark.parametrize("name,shape,cfg", MODES, ids=[m[0] for m in MODES])
def test_bias_act_parity(name, shape, cfg, act):
    M, N, K = shape
    for dtype in ("f16", "bf16"):
        A, B = inputs.make_operands(M, N, K, dtype)
        bias = (torch.randn(N, generator=torch.Generator().manual_seed(N)) * 4).float()
        C = pu.run_gpu_epilogue(A, B, dtype, cfg, bias, act)
        _check(A, B, dtype, C, bias.numpy(), act, "%s act=%d %s" % (name, act, dtype))


def test_no_bias_with_activation():
    A, B = inputs.make_operands(256, 128, 512, "f16")
    C = pu.run_gpu_epilogue(A, B, "f16", {"block_n": 128}, None, oracle.ACT_RELU)
    _check(A, B, "f16", C, None, oracle.ACT_RELU, "relu without bias")
    assert torch.all(C >= 0)


def test_k_zero_gives_act_of_bias():
    bias = torch.linspace(-3, 3, 64).float()
    A = torch.empty(5, 0, dtype=torch.float16)
    B = torch.empty(64, 0, dtype=torch.float16)
    C = pu.run_gpu_epilogue(A, B, "f16", None, bias, oracle.ACT_GELU)
    want = oracle.epilogue(np.zeros((5, 64)), bias.numpy(), oracle.ACT_GELU)
    assert np.allclose(C.float().cpu().numpy(), want, rtol=2e-3, atol=1e-3)


def test_ffn_shape_gelu_sampled():
    w = workloads.FFN_BF16
    A, B = inputs.make_operands(w.M, w.N, w.K, w.dtype, w.a_scale, w.b_scale)
    bias = (torch.randn(w.N, generator=torch.Generator().manual_seed(7)) * 0.5).float()
    C = pu.run_gpu_epilogue(A, B, w.dtype, None, bias, oracle.ACT_GELU)
    rows, cols = inputs.sample_positions(w.M, w.N, 4096, 11)
    _check(A, B, w.dtype, C, bias.numpy(), oracle.ACT_GELU, "ffn gelu", rows.numpy(), cols.numpy())


@pytest.mark.parametrize("shape,cfg", [((2560, 1280, 512), {"block_n": 64}),
                                       ((4096, 2048, 256), {"block_n": 256})],
                         ids=["one_sm_64", "one_sm_256"])
def test_multi_tile_epilogue_sampled(shape, cfg):
    """One-SM CTAs that run several tiles each (the bias of a tile's first chunk is
    fetched while the previous tile is still being stored), sampled."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "f16")
    bias = (torch.randn(N, generator=torch.Generator().manual_seed(3)) * 2).float()
    for act in (oracle.ACT_GELU, oracle.ACT_SILU):
        C = pu.run_gpu_epilogue(A, B, "f16", cfg, bias, act)
        rows, cols = inputs.sample_positions(M, N, 4096, 5 + act)
        _check(A, B, "f16", C, bias.numpy(), act, "multi-tile act=%d" % act, rows.numpy(),
               cols.numpy())


def test_rejects_bad_epilogue_arguments(gemm_lib):
    g = gemm_lib
    A = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    bias = torch.zeros(80, dtype=torch.float32, device="cuda")
    with g.Plan(64, 64, 64, "f16") as p:
        with pytest.raises(g.GemmError) as e:
            g.gemm_run_bias_act(p.handle, A, A, C, bias[1:].data_ptr(), 1)
        assert e.value.status == 3
        with pytest.raises(g.GemmError) as e:
            g.gemm_run_bias_act(p.handle, A, A, C, bias, 7)
        assert e.value.status == 1
    Ai = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    Ci = torch.zeros(64, 64, dtype=torch.int32, device="cuda")
    with g.Plan(64, 64, 64, "i8") as p:
        with pytest.raises(g.GemmError) as e:
            g.gemm_run_bias_act(p.handle, Ai, Ai, Ci, bias, 0)
        assert e.value.status == 2
