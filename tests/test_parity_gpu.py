"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small and medium shapes are checked on every element (they span several tiles
and ragged tails in M, N and K, and every kernel variant: tile widths 64/128/256,
split-K); the full-size workloads are checked on >= 4096 seeded sampled
elements (corners and tile-edge rows/columns included) in the configuration the
benchmark runs.
"""
import numpy as np
import pytest
import torch

from dense_gemm_hgemm_gb300 import inputs, workloads

import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(gemm_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gemm_lib


# --------------------------------------------------------------------------- smallest first

def test_single_tile_f16():
    A, B = inputs.make_operands(128, 64, 64, "f16")
    C = pu.run_gpu(A, B, "f16", {"block_n": 64})
    pu.check_full(A, B, "f16", C, "128x64x64")


def test_exact_small_integers_bit_exact():
    """Entries in {-2..2}: every partial sum is an integer <= 4096, so fp32
    accumulation is exact and the fp16 output equals the integer result."""
    M, N, K = 256, 512, 1024
    for dtype in ("f16", "bf16"):
        A = inputs.small_integers(M, K, -2, 2, dtype, 31)
        B = inputs.small_integers(N, K, -2, 2, dtype, 32)
        want = (A.to(torch.int64) @ B.to(torch.int64).T)
        for bn in (64, 128, 256):
            C = pu.run_gpu(A, B, dtype, {"block_n": bn})
            got = C.cpu().to(torch.float64)
            rep = want.to(inputs.TORCH_DTYPE[dtype]).to(torch.float64)   # |want| > 256 rounds in bf16
            assert torch.equal(got, rep), (dtype, bn)


SMALL_SHAPES = [
    (1, 8, 8), (64, 64, 64), (128, 128, 64), (130, 72, 200), (257, 520, 264), (300, 264, 1000),
    (64, 4096, 64), (128, 2048, 128), (384, 768, 512),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_full_parity_small(shape, bn, dtype):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dtype)
    C = pu.run_gpu(A, B, dtype, {"block_n": bn})
    pu.check_full(A, B, dtype, C, "%s bn=%d %s" % (shape, bn, dtype))


@pytest.mark.parametrize("split", [2, 3, 7])
@pytest.mark.parametrize("shape", [(128, 128, 4096), (200, 136, 1000), (64, 64, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_k_parity_and_determinism(shape, split):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "f16")
    C1 = pu.run_gpu(A, B, "f16", {"block_n": 64, "split_k": split}, repeats=3)
    pu.check_full(A, B, "f16", C1, "split %d %s" % (split, shape))
    C2 = pu.run_gpu(A, B, "f16", {"block_n": 64, "split_k": split})
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8"])
@pytest.mark.parametrize("split", [2, 4, 8])
@pytest.mark.parametrize("shape", [(128, 128, 4096), (200, 136, 1024), (64, 64, 2048),
                                   (384, 264, 512)], ids=lambda s: "x".join(map(str, s)))
def test_cluster_split_k_parity_and_determinism(shape, split, dtype):
    """Split-K whose slices form one thread-block cluster per tile, reduced in
    distributed shared memory in slice order."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dtype)
    for bn in ((64, 128) if dtype == "i8" else (64, 256)):
        cfg = {"block_n": bn, "split_k": split, "split_mode": 1}
        C1 = pu.run_gpu(A, B, dtype, cfg, repeats=3)
        pu.check_full(A, B, dtype, C1, "cluster split %d bn=%d %s %s" % (split, bn, shape, dtype))
        C2 = pu.run_gpu(A, B, dtype, cfg)
        assert torch.equal(C1.view(torch.int16) if dtype != "i8" else C1,
                           C2.view(torch.int16) if dtype != "i8" else C2)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("shape", [(256, 128, 64), (64, 136, 128), (300, 264, 1000),
                                   (1000, 520, 1024), (2048, 1536, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_kernel_parity(shape, bn, dtype):
    """256-row tiles on an SM pair (tcgen05 cta_group::2): ragged M (one CTA of
    the pair entirely beyond M), ragged N, several tiles per pair."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dtype)
    C = pu.run_gpu(A, B, dtype, {"block_n": bn, "cta_pair": 1}, repeats=2)
    pu.check_full(A, B, dtype, C, "pair bn=%d %s %s" % (bn, shape, dtype))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8"])
@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("shape", [(256, 128, 1024), (300, 264, 1000), (1000, 520, 4096),
                                   (64, 136, 640)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_cluster_split_k_parity_and_determinism(shape, split, dtype):
    """SM pairs with K sliced across the pairs of one cluster (2 * split CTAs),
    reduced in distributed shared memory in slice order: ragged M (the peer's
    half beyond M), ragged N and K, uneven last slice."""
    M, N, K = shape
    if dtype == "i8":
        K = -(-K // 16) * 16                  # int8 rows must be whole 16-byte groups
    A, B = inputs.make_operands(M, N, K, dtype)
    for bn in ((128,) if dtype == "i8" else (128, 256)):
        cfg = {"block_n": bn, "cta_pair": 1, "split_k": split, "split_mode": 1}
        C1 = pu.run_gpu(A, B, dtype, cfg, repeats=2)
        pu.check_full(A, B, dtype, C1, "pair split %d bn=%d %s %s" % (split, bn, shape, dtype))
        C2 = pu.run_gpu(A, B, dtype, cfg)
        assert torch.equal(C1.view(torch.int16) if dtype != "i8" else C1,
                           C2.view(torch.int16) if dtype != "i8" else C2)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "i8"])
@pytest.mark.parametrize("shape", [(64, 4096, 64), (130, 72, 208), (257, 520, 1040)],
                         ids=lambda s: "x".join(map(str, s)))
def test_direct_store_epilogue_parity(shape, dtype):
    """The per-thread 16-byte store epilogue (instead of TMA stores)."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dtype)
    for bn in ((64, 128) if dtype == "i8" else (64, 128, 256)):
        C = pu.run_gpu(A, B, dtype, {"block_n": bn, "direct_store": 1})
        pu.check_full(A, B, dtype, C, "direct store bn=%d %s %s" % (bn, shape, dtype))


def test_default_config_headline_shapes():
    for w in (workloads.SKINNY, workloads.HEADLINE_SWEEP):
        A, B = inputs.make_operands(w.M, w.N, w.K, w.dtype, w.a_scale, w.b_scale)
        C = pu.run_gpu(A, B, w.dtype)
        pu.check_full(A, B, w.dtype, C, w.name)


@pytest.mark.parametrize("shape,dtype", [((2104, 2104, 2104), "f16"), ((1000, 3000, 4160), "bf16"),
                                         ((2112, 2104, 2112), "i8")])
def test_cost_model_shapes_sampled(shape, dtype):
    """Shapes outside the measured table run the cost model's configuration (here
    SM pairs, 256- or 128-wide, with ragged edges), checked on sampled elements."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, dtype)
    C = pu.run_gpu(A, B, dtype)
    pu.check_sampled(A, B, dtype, C, where="cost model %s %s" % (shape, dtype))


def _random_shapes(n, seed):
    import random
    rnd = random.Random(seed)
    out = []
    for _ in range(n):
        dt = rnd.choice(("f16", "bf16", "i8"))
        M = rnd.randint(1, 3000)
        N = rnd.randint(1, 500) * 4 if dt == "i8" else rnd.randint(1, 300) * 8
        K = rnd.randint(1, 200) * (16 if dt == "i8" else 8)
        out.append((M, N, K, dt))
    return out


@pytest.mark.parametrize("M,N,K,dtype", _random_shapes(12, 5))
def test_random_shapes_cost_model_sampled(M, N, K, dtype):
    """Seeded random shapes with the configuration the library chooses, sampled."""
    A, B = inputs.make_operands(M, N, K, dtype)
    C = pu.run_gpu(A, B, dtype)
    pu.check_sampled(A, B, dtype, C, count=2048, where="random %dx%dx%d %s" % (M, N, K, dtype))


# --------------------------------------------------------------------------- int8 -> int32

@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("shape", [(128, 64, 64), (130, 72, 208), (257, 520, 1040), (64, 4096, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_int8_bit_exact_small(shape, bn):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "i8")
    C = pu.run_gpu(A, B, "i8", {"block_n": bn})
    pu.check_full(A, B, "i8", C, "i8 %s bn=%d" % (shape, bn))


def test_int8_extremes_k4096():
    """All -128 (largest products) and mixed 127/-128 at K=4096: |sum| up to 2^26,
    exact only if every fp32 chunk partial stays exact."""
    K = 4096
    A = torch.full((256, K), -128, dtype=torch.int8)
    B = torch.full((192, K), -128, dtype=torch.int8)
    B[1::2] = 127
    C = pu.run_gpu(A, B, "i8", {"block_n": 64}).cpu()
    assert torch.all(C[:, 0::2] == K * 16384)
    assert torch.all(C[:, 1::2] == -128 * 127 * K)
    pu.check_full(A, B, "i8", pu.run_gpu(A, B, "i8", {"block_n": 128}), "i8 extremes")


@pytest.mark.parametrize("shape", [(256, 128, 1024), (300, 264, 1040), (1000, 520, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
def test_int8_pair_kernel_bit_exact(shape):
    """Integer mode on an SM pair: chunked exact fp32 accumulation drained to int32."""
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "i8")
    C = pu.run_gpu(A, B, "i8", {"block_n": 128, "cta_pair": 1}, repeats=2)
    pu.check_full(A, B, "i8", C, "i8 pair %s" % (shape,))


@pytest.mark.parametrize("cfg", [{"block_n": 64}, {"block_n": 128}, {"block_n": 128, "cta_pair": 1}],
                         ids=["bn64", "bn128", "pair"])
def test_int8_small_addend_at_top_of_range(cfg):
    """Per 1024-long K chunk: 1023 products of 2^14 then one product of 1, i.e. a
    partial sum of 2^24 - 2^14 + 1 that needs all 24 significand bits of the fp32
    accumulator (a narrower internal adder drops the +1); other rows mix signs."""
    K = 4096
    A = torch.full((256, K), -128, dtype=torch.int8)
    B = torch.full((128, K), -128, dtype=torch.int8)
    for c in range(K // 1024):
        A[:, c * 1024 + 1023] = 1
        B[:, c * 1024 + 1023] = 1
    A[1::2, ::2] = 127                       # odd rows: alternating large mixed-sign products
    C = pu.run_gpu(A, B, "i8", cfg).cpu()
    assert torch.all(C[0::2] == 4 * (1023 * 16384 + 1))
    pu.check_full(A, B, "i8", C, "small addend %s" % cfg)


def test_int8_pair_kernel_extremes():
    K = 4096
    A = torch.full((384, K), -128, dtype=torch.int8)
    B = torch.full((256, K), -128, dtype=torch.int8)
    B[1::2] = 127
    C = pu.run_gpu(A, B, "i8", {"block_n": 128, "cta_pair": 1}).cpu()
    assert torch.all(C[:, 0::2] == K * 16384)
    assert torch.all(C[:, 1::2] == -128 * 127 * K)


def test_int8_split_k():
    A, B = inputs.make_operands(128, 128, 4096, "i8")
    C = pu.run_gpu(A, B, "i8", {"block_n": 64, "split_k": 4})
    pu.check_full(A, B, "i8", C, "i8 split-K")


# --------------------------------------------------------------------------- edges

def test_k_zero_writes_zeros():
    A = torch.empty(70, 0, dtype=torch.float16)
    B = torch.empty(48, 0, dtype=torch.float16)
    C = torch.full((70, 48), 7.0, dtype=torch.float16, device="cuda")
    pu.run_gpu(A, B, "f16", out=C)
    assert torch.all(C == 0)


def test_empty_m_is_a_no_op():
    A = torch.empty(0, 64, dtype=torch.float16)
    B = torch.ones(32, 64, dtype=torch.float16)
    C = torch.empty(0, 32, dtype=torch.float16, device="cuda")
    pu.run_gpu(A, B, "f16", out=C)


def test_guard_bands_untouched():
    """C inside a larger buffer: the bytes before and after C stay unchanged."""
    M, N, K = 200, 136, 512
    A, B = inputs.make_operands(M, N, K, "bf16")
    pad = 4096
    buf = torch.full((pad * 2 + M * N,), 3.5, dtype=torch.bfloat16, device="cuda")
    C = buf[pad:pad + M * N].view(M, N)
    pu.run_gpu(A, B, "bf16", {"block_n": 256}, out=C)
    assert torch.all(buf[:pad] == 3.5) and torch.all(buf[pad + M * N:] == 3.5)
    pu.check_full(A, B, "bf16", C, "guarded")


def test_run_rejects_misaligned_pointers():
    import dense_gemm_hgemm_gb300 as g
    A = torch.zeros(64 * 64 + 8, dtype=torch.float16, device="cuda")
    B = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    with g.Plan(64, 64, 64, "f16") as p:
        with pytest.raises(g.GemmError) as e:
            p.run(A[1:].data_ptr(), B, C)
        assert e.value.status == 3


# --------------------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("w", [workloads.SQUARE_8192, workloads.FFN_BF16, workloads.INT8_4096],
                         ids=lambda w: w.name)
def test_full_size_sampled(w):
    A, B = inputs.make_operands(w.M, w.N, w.K, w.dtype, w.a_scale, w.b_scale)
    C = pu.run_gpu(A, B, w.dtype, repeats=2)
    pu.check_sampled(A, B, w.dtype, C, count=4096, where=w.name)
    del C
    torch.cuda.empty_cache()
