"""Operand storages other than TN (M/N-contiguous tiles, M/N-major descriptors).

The math is the TN oracle's: the test stores the same logical operands
transposed (B as K x N for NN, A as K x M for TT, both for NT) and compares
with the oracle run on the untransposed operands."""
import pytest

from dense_gemm_hgemm_gb300 import inputs

import parity_util as pu

pytestmark = pytest.mark.gpu

CONFIGS = [
    ("bn64", {"block_n": 64}),
    ("bn128", {"block_n": 128}),
    ("bn256", {"block_n": 256}),
    ("pair128", {"block_n": 128, "cta_pair": 1}),
    ("pair256", {"block_n": 256, "cta_pair": 1}),
    ("split_ws", {"block_n": 64, "split_k": 3}),
    ("split_cluster", {"block_n": 128, "split_k": 4, "split_mode": 1}),
    ("pair_split", {"block_n": 256, "cta_pair": 1, "split_k": 2, "split_mode": 1}),
    ("multicast2", {"block_n": 64, "multicast": 2}),
]
SHAPES = [(136, 72, 200), (384, 264, 512), (1000, 520, 1024)]


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
@pytest.mark.parametrize("name,cfg", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_layout_parity(layout, name, cfg):
    for dtype in ("f16", "bf16"):
        for M, N, K in SHAPES:
            A, B = inputs.make_operands(M, N, K, dtype)
            C = pu.run_gpu_layout(A, B, dtype, cfg, layout)
            pu.check_full(A, B, dtype, C, "%s %s %s %s" % (layout, name, (M, N, K), dtype))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
@pytest.mark.parametrize("cfg", [{"block_n": 64}, {"block_n": 128, "cta_pair": 1}], ids=["bn64", "pair"])
def test_layout_int8_bit_exact(layout, cfg):
    for M, N, K in ((144, 80, 208), (512, 272, 1040)):
        A, B = inputs.make_operands(M, N, K, "i8")
        C = pu.run_gpu_layout(A, B, "i8", cfg, layout)
        pu.check_full(A, B, "i8", C, "i8 %s %s" % (layout, (M, N, K)))


@pytest.mark.parametrize("layout", ["NN", "TT", "NT"])
def test_layout_default_config(layout):
    A, B = inputs.make_operands(2048, 1024, 512, "f16")
    C = pu.run_gpu_layout(A, B, "f16", None, layout)
    pu.check_sampled(A, B, "f16", C, count=2048, where="default %s" % layout)
