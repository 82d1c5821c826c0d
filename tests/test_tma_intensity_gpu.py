"""The TMA load-mode x intensity experiment: every mode computes the same
elementwise fma chain, bit-exact against the oracle's single-rounding fmaf."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

N = 4_194_304          # the page's workload: 4 Mi floats, 2048 x 2048 view, 64 tiles per block
A_COEF, B_COEF = 0.999, 0.001


@pytest.fixture(scope="module")
def data():
    g = torch.Generator().manual_seed(2024)
    return torch.randn(N, generator=g, dtype=torch.float32)


@pytest.mark.parametrize("iters", [0, 1, 8, 64])
@pytest.mark.parametrize("mode", ["sync", "bulk1d", "tensor2d", "pipe2"])
def test_modes_bit_exact(gemm_lib, data, mode, iters):
    x = data.cuda()
    y = torch.full_like(x, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gemm_lib.tma_intensity_run(mode, iters, A_COEF, B_COEF, x, y, 2048, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.fma_chain(data.numpy(), iters, np.float32(A_COEF), np.float32(B_COEF))
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), mode


def test_rejects_bad_sizes(gemm_lib):
    x = torch.zeros(65536 + 1024, device="cuda")
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.tma_intensity_run("sync", 1, 1.0, 0.0, x, x)
    x = torch.zeros(65536, device="cuda")
    with pytest.raises(gemm_lib.GemmError):
        gemm_lib.tma_intensity_run("tensor2d", 1, 1.0, 0.0, x, x, cols=48)
