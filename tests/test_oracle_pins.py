"""Pins for the CPU oracle: checks against facts the mathematics fixes.

Each test is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong exponent bias in the
decoders, a missing wrap) fails at least one of them.  ``test_oracle_mutants``
plants such mistakes in a copy of the oracle source and checks that the pins
catch them.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

from dense_gemm_hgemm_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _fmt(dtype):
    return 0 if dtype == "f16" else 1


# ---------------------------------------------------------------------------
# decoders: exhaustive over all 65,536 patterns
# ---------------------------------------------------------------------------

def test_f16_decoder_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.decode(bits, 0)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle_mod.decode(bits.astype(np.uint16), 1)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decoder_landmarks(oracle_mod):
    # values fixed by the two formats' definitions
    f16 = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
           0x3555: 0.333251953125}
    for b, v in f16.items():
        assert oracle_mod.decode(np.array([b], np.uint16), 0)[0] == v
    bf16 = {0x3F80: 1.0, 0xC000: -2.0, 0x7F7F: 3.3895313892515355e38, 0x0001: 2.0 ** -133,
            0x3EAB: 0.333984375}
    for b, v in bf16.items():
        assert oracle_mod.decode(np.array([b], np.uint16), 1)[0] == v


# ---------------------------------------------------------------------------
# brute force on tiny inputs against an independent integer formulation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_brute_force_tiny(oracle_mod, dtype):
    sizes = (1, 2, 3, 5)
    seed = 11
    for M in sizes:
        for N in sizes:
            for K in sizes:
                seed += 1
                A = inputs.small_integers(M, K, -3, 3, dtype, seed)
                B = inputs.small_integers(N, K, -3, 3, dtype, seed + 1000)
                got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), _fmt(dtype))
                Ai = A.to(torch.int64).numpy()
                Bi = B.to(torch.int64).numpy()
                want = Ai @ Bi.T
                assert got.shape == (M, N)
                assert np.array_equal(got, want.astype(np.float64)), (M, N, K)


def test_brute_force_tiny_i8(oracle_mod):
    seed = 77
    for M in (1, 2, 3, 5):
        for N in (1, 2, 3, 5):
            for K in (1, 2, 3, 5, 16):
                seed += 1
                g = torch.Generator().manual_seed(seed)
                A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8).numpy()
                B = torch.randint(-128, 128, (N, K), generator=g, dtype=torch.int8).numpy()
                c64, c32 = oracle_mod.gemm_tn_i8(A, B)
                want = A.astype(np.int64) @ B.astype(np.int64).T
                assert np.array_equal(c64, want)
                assert np.array_equal(c32, want.astype(np.int32))


def test_python_loop_formulation(oracle_mod):
    """A pure-Python triple loop over exact rationals on a ragged 3x4x5 case."""
    from fractions import Fraction
    A = inputs.make_operands(3, 4, 5, "f16")[0]
    B = inputs.make_operands(4, 3, 5, "f16")[0]
    a = [[Fraction(float(x)) for x in row] for row in A.float().tolist()]
    b = [[Fraction(float(x)) for x in row] for row in B.float().tolist()]
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), 0)
    for i in range(3):
        for j in range(4):
            exact = sum(a[i][k] * b[j][k] for k in range(5))
            assert abs(Fraction(got[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def test_empty_sum_is_zero(oracle_mod):
    A = np.zeros((3, 0), np.uint16)
    B = np.zeros((4, 0), np.uint16)
    assert np.array_equal(oracle_mod.gemm_tn_half(A, B, 0), np.zeros((3, 4)))
    c64, c32 = oracle_mod.gemm_tn_i8(np.zeros((2, 0), np.int8), np.zeros((5, 0), np.int8))
    assert np.array_equal(c64, np.zeros((2, 5))) and np.array_equal(c32, np.zeros((2, 5)))


# ---------------------------------------------------------------------------
# identity, permutation, rank-1 closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_identity_gives_transpose(oracle_mod, dtype):
    K, N = 48, 37
    A = torch.eye(K, dtype=inputs.TORCH_DTYPE[dtype])
    B = inputs.make_operands(K, N, K, dtype)[1]
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), _fmt(dtype))
    want = B.double().numpy().T          # ref[i][j] = B[j][i]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_permutation_rows(oracle_mod, dtype):
    K, N = 40, 29
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(5))
    A = torch.zeros(K, K, dtype=inputs.TORCH_DTYPE[dtype])
    A[torch.arange(K), perm] = 1
    B = inputs.make_operands(K, N, K, dtype)[1]
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), _fmt(dtype))
    want = B.double().numpy()[:, perm.numpy()].T   # ref[i][j] = B[j][perm[i]]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_rank1_closed_form(oracle_mod, dtype):
    M, N, K = 13, 17, 64
    g = torch.Generator().manual_seed(9)
    u = torch.randint(-4, 5, (M,), generator=g).double()
    v = torch.randint(-4, 5, (N,), generator=g).double()
    x = 2.0 ** torch.randint(-3, 4, (K,), generator=g).double()
    y = torch.randint(-3, 4, (K,), generator=g).double()
    td = inputs.TORCH_DTYPE[dtype]
    A = (u[:, None] * x[None, :]).to(td)
    B = (v[:, None] * y[None, :]).to(td)
    assert torch.equal(A.double(), u[:, None] * x[None, :])   # inputs exact in the format
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), _fmt(dtype))
    want = (u[:, None] * v[None, :] * float((x * y).sum())).numpy()
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exact_small_integers(oracle_mod, dtype):
    M, N, K = 40, 24, 1024
    A = inputs.small_integers(M, K, -2, 2, dtype, 21)
    B = inputs.small_integers(N, K, -2, 2, dtype, 22)
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), _fmt(dtype))
    want = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    assert np.array_equal(got, want.astype(np.float64))


def test_asymmetric_operands_not_swapped(oracle_mod):
    """C = A B^T, not B A^T or A^T B: distinct M, N, K and a non-symmetric product."""
    A = torch.tensor([[1, 2, 3]], dtype=torch.float16)            # 1 x 3
    B = torch.tensor([[1, 0, 0], [0, 0, 2]], dtype=torch.float16)  # 2 x 3
    got = oracle_mod.gemm_tn_half(_bits(A), _bits(B), 0)
    assert np.array_equal(got, np.array([[1.0, 6.0]]))


# ---------------------------------------------------------------------------
# int8 extremes and the wrap to int32
# ---------------------------------------------------------------------------

def test_i8_extremes(oracle_mod):
    K = 4096
    A = np.full((3, K), -128, np.int8)
    B = np.full((2, K), -128, np.int8)
    c64, c32 = oracle_mod.gemm_tn_i8(A, B)
    assert np.all(c64 == K * 16384) and np.all(c32 == 2 ** 26)
    B2 = np.full((2, K), 127, np.int8)
    c64, c32 = oracle_mod.gemm_tn_i8(A, B2)
    assert np.all(c64 == -128 * 127 * K) and np.all(c32 == -128 * 127 * K)
    # alternating signs cancel exactly
    A3 = np.tile(np.array([127, -128], np.int8), (1, K // 2))
    B3 = np.full((1, K), 1, np.int8)
    c64, _ = oracle_mod.gemm_tn_i8(A3, B3)
    assert c64[0, 0] == (127 - 128) * (K // 2)


def test_i8_wraps_modulo_2_32(oracle_mod):
    K = 131072                      # 2^17 * 2^14 = 2^31 overflows int32 by one
    A = np.full((1, K + 1), -128, np.int8)
    B = np.full((1, K + 1), -128, np.int8)
    A[0, K] = 0
    c64, c32 = oracle_mod.gemm_tn_i8(A, B)
    assert c64[0, 0] == 2 ** 31 and c32[0, 0] == -2 ** 31
    A[0, K] = -128
    c64, c32 = oracle_mod.gemm_tn_i8(A, B)
    assert c64[0, 0] == 2 ** 31 + 2 ** 14 and c32[0, 0] == -2 ** 31 + 2 ** 14


# ---------------------------------------------------------------------------
# sampled evaluation = the same definition at chosen positions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_sampled_matches_brute_force(oracle_mod, dtype):
    M, N, K = 9, 11, 7
    A = inputs.small_integers(M, K, -3, 3, dtype, 1)
    B = inputs.small_integers(N, K, -3, 3, dtype, 2)
    want = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    rows, cols = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = oracle_mod.gemm_tn_half_sampled(_bits(A), _bits(B), _fmt(dtype), rows.ravel(),
                                          cols.ravel())
    assert np.array_equal(got.reshape(M, N), want.astype(np.float64))


def test_sampled_i8_matches_brute_force(oracle_mod):
    g = torch.Generator().manual_seed(3)
    A = torch.randint(-128, 128, (6, 33), generator=g, dtype=torch.int8).numpy()
    B = torch.randint(-128, 128, (5, 33), generator=g, dtype=torch.int8).numpy()
    want = A.astype(np.int64) @ B.astype(np.int64).T
    rows, cols = np.meshgrid(np.arange(6), np.arange(5), indexing="ij")
    o64, o32 = oracle_mod.gemm_tn_i8_sampled(A, B, rows.ravel(), cols.ravel())
    assert np.array_equal(o64.reshape(6, 5), want)
    assert np.array_equal(o32.reshape(6, 5), want.astype(np.int32))


def test_sampled_rejects_out_of_range(oracle_mod):
    A = np.zeros((2, 4), np.uint16)
    with pytest.raises(RuntimeError):
        oracle_mod.gemm_tn_half_sampled(A, A, 0, [0, 2], [0, 0])


# ---------------------------------------------------------------------------
# statistics of the seeded N(0,1) workload
# ---------------------------------------------------------------------------

def test_variance_of_randn_product(oracle_mod):
    M, N, K = 64, 64, 256
    A, B = inputs.make_operands(M, N, K, "f16")
    C = oracle_mod.gemm_tn_half(_bits(A), _bits(B), 0)
    var = C.var()
    assert abs(var / K - 1.0) < 0.10, var / K
    assert abs(C.mean()) < 0.1 * np.sqrt(K)


def test_worked_example_golden(oracle_mod):
    """The hand-worked fixture in tests/golden/ (derivation written in the file)."""
    path = os.path.join(HERE, "golden", "gemm_tn_worked_example.txt")
    blocks = {}
    cur = None
    for line in open(path, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.endswith(":"):
            cur = line[:-1]
            blocks[cur] = []
        else:
            blocks[cur].append([float(x) for x in line.split()])
    A = torch.tensor(blocks["A"], dtype=torch.float16)
    B = torch.tensor(blocks["B"], dtype=torch.float16)
    want = np.array(blocks["C"])
    assert np.array_equal(oracle_mod.gemm_tn_half(_bits(A), _bits(B), 0), want)
    assert np.array_equal(oracle_mod.gemm_tn_half(_bits(A.bfloat16()), _bits(B.bfloat16()), 1), want)


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (mutants of the oracle source, built on the CPU)
# ---------------------------------------------------------------------------

MUTANTS = {
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) s += Ad", "for (int64_t k = 0; k < K - 1; ++k) s += Ad"),
    "transposed_B": ("Bd[j * K + k]", "Bd[k * N + j]"),
    "wrong_sign": ("s += Ad[i * K + k] * Bd[j * K + k]", "s -= Ad[i * K + k] * Bd[j * K + k]"),
    "f16_bias": ("ldexp((double)(m | 0x400), e - 25)", "ldexp((double)(m | 0x400), e - 24)"),
    "bf16_subnormal": ("ldexp((double)m, -133)", "ldexp((double)m, -126)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_oracle_mutants_are_caught(tmp_path, name):
    import ctypes
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "gemm_oracle.c")).read()
    old, new = MUTANTS[name]
    assert old in src
    so = tmp_path / "mut.so"
    (tmp_path / "mut.c").write_text(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-shared", "-fPIC", str(tmp_path / "mut.c"),
                    "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_gemm_tn_half.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_decode.argtypes = [p, p, i64, ctypes.c_int]

    def gemm(A, B, fmt):
        A, B = np.ascontiguousarray(A), np.ascontiguousarray(B)
        C = np.empty((A.shape[0], B.shape[0]))
        lib.oracle_gemm_tn_half(A.ctypes.data, B.ctypes.data, C.ctypes.data, A.shape[0],
                                B.shape[0], A.shape[1], fmt, 1)
        return C

    caught = False
    # the pin set, re-run against the mutant
    for fmt, td in ((0, torch.float16), (1, torch.bfloat16)):
        A = inputs.small_integers(5, 7, -3, 3, "f16" if fmt == 0 else "bf16", 1)
        B = inputs.small_integers(6, 7, -3, 3, "f16" if fmt == 0 else "bf16", 2)
        want = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
        caught |= not np.array_equal(gemm(_bits(A), _bits(B), fmt), want)
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        out = np.empty(65536)
        lib.oracle_decode(bits.ctypes.data, out.ctypes.data, 65536, fmt)
        with np.errstate(invalid="ignore"):
            ref = bits.view(np.float16).astype(np.float64) if fmt == 0 else \
                (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ok = np.isnan(ref)
        caught |= not np.array_equal(out[~ok], ref[~ok])
        Ae = torch.eye(7, dtype=td)
        Be = inputs.make_operands(7, 7, 7, "f16" if fmt == 0 else "bf16")[1]
        caught |= not np.array_equal(gemm(_bits(Ae), _bits(Be), fmt), Be.double().numpy().T)
    assert caught, name


# ---------------------------------------------------------------------------
# fused epilogue act(C + bias): closed forms
# ---------------------------------------------------------------------------

def test_epilogue_closed_forms(oracle_mod):
    C = np.array([[0.0, 1.0, -1.0, 2.0]])
    bias = np.array([0.0, 0.0, 0.0, -2.0], np.float32)
    assert np.array_equal(oracle_mod.epilogue(C, bias, 0), [[0.0, 1.0, -1.0, 0.0]])
    assert np.array_equal(oracle_mod.epilogue(C, None, 1), [[0.0, 1.0, 0.0, 2.0]])
    g = oracle_mod.epilogue(C, None, 2)[0]
    # GELU(x) = x * Phi(x): Phi(0) = 1/2, Phi(1) = 0.8413447460685429 (standard normal table)
    assert g[0] == 0.0 and abs(g[1] - 0.8413447460685429) < 1e-15
    assert abs(g[2] - (-1.0) * (1 - 0.8413447460685429)) < 1e-15
    s = oracle_mod.epilogue(C, None, 3)[0]
    # SiLU(x) = x * sigmoid(x): sigmoid(1) = e / (1 + e)
    assert s[0] == 0.0 and abs(s[1] - np.e / (1 + np.e)) < 1e-15
    assert abs(s[2] - (-1.0) / (1 + np.e)) < 1e-15      # sigmoid(-1) = 1/(1+e)


def test_epilogue_bias_is_per_column(oracle_mod):
    C = np.zeros((3, 4))
    bias = np.array([1, -2, 3, -4], np.float32)
    out = oracle_mod.epilogue(C, bias, 1)
    assert np.array_equal(out, np.tile([[1.0, 0.0, 3.0, 0.0]], (3, 1)))
    vals = oracle_mod.epilogue_sampled(np.zeros(4), [3, 2, 1, 0], bias, 0)
    assert np.array_equal(vals, [-4.0, 3.0, -2.0, 1.0])


def test_epilogue_symmetries(oracle_mod):
    x = np.linspace(-6, 6, 241)[None, :]
    g = oracle_mod.epilogue(x, None, 2)[0]
    # GELU(x) - GELU(-x) = x  (since Phi(x) + Phi(-x) = 1)
    assert np.allclose(g - g[::-1], x[0], atol=1e-14, rtol=0)
    s = oracle_mod.epilogue(x, None, 3)[0]
    assert np.allclose(s - s[::-1], x[0], atol=1e-14, rtol=0)   # sigmoid(x) + sigmoid(-x) = 1
    with pytest.raises(RuntimeError):
        oracle_mod.epilogue(x, None, 9)


# ---------------------------------------------------------------------------
# fma chain of the TMA intensity experiment
# ---------------------------------------------------------------------------

def test_fma_chain_closed_form_and_single_rounding(oracle_mod):
    x = np.array([0.0, 1.0, -2.0, 3.5], np.float32)
    assert np.array_equal(oracle_mod.fma_chain(x, 0, 0.5, 1.0), x)
    # a = 1/2, b = 1: exact in fp32, y_k = 2 + (x - 2) / 2^k
    for k in (1, 2, 5):
        assert np.array_equal(oracle_mod.fma_chain(x, k, 0.5, 1.0),
                              (2.0 + (x.astype(np.float64) - 2.0) / 2 ** k).astype(np.float32))
    # fused: fma(1 + 2^-23, 1 - 2^-23, -1) = -2^-46 exactly (a separate multiply rounds it to 0)
    one_p = np.float32(1 + 2 ** -23)
    y = oracle_mod.fma_chain(np.array([one_p], np.float32), 1, float(np.float32(1 - 2 ** -23)), -1.0)
    assert y[0] == np.float32(-(2.0 ** -46))
