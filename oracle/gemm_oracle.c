/*
 * gemm_oracle.c -- plain, slow CPU oracle for the TN GEMM  C = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's timed CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (the definition, written out with no blocking or reordering):
 *
 *   half-precision operands (HGEMM, "row-major A and col-major B"):
 *       C[i][j] = sum_{k=0}^{K-1} double(A[i][k]) * double(B[j][k])        (fp64 accumulation)
 *   int8 operands (the "FP16/INT8 switch" of the same kernel family):
 *       C[i][j] = sum_{k=0}^{K-1} int64(A[i][k]) * int64(B[j][k])          (int64 accumulation)
 *       and the int32 result is that sum reduced modulo 2^32 (two's complement).
 *
 *   Sources: "RL驱动CUDA L2 GEMM内核自动调优：A100/H100 tile size与融合优化"
 *   (blog.hotdry.top, 2025-12-05), paragraph on tile size / data layout (A row-major,
 *   B column-major, i.e. both operands contiguous along K), paragraph on multi-precision
 *   adaptation (FP16 / INT8), and its correctness paragraph (randn inputs, relative
 *   error against a library GEMM).  The pages leave the accumulator precision open;
 *   the oracle uses fp64 (int64 for int8) so that its own rounding is far below the
 *   tolerance the GPU result is held to.
 *
 * Layouts: A is M x K row-major, B is N x K row-major, C is M x N row-major.
 * Half-precision inputs arrive as raw 16-bit patterns and are decoded here from the
 * IEEE 754 binary16 definition and the bfloat16 definition (the upper half of an
 * IEEE 754 binary32), never through a GPU or library conversion.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (the contraction flag keeps
 * every multiply and add separately rounded in fp64, the same on x86-64 and aarch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(m | 0x400), e - 25);    /* (1 + m/2^10) * 2^(e-15)      */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b)
{
    const int sign = (b >> 15) & 1;
    const int e = (b >> 7) & 0xff;
    const int m = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -133);                /* subnormal: m * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(m | 0x80), e - 134);    /* (1 + m/2^7) * 2^(e-127)      */
    }
    return sign ? -v : v;
}

static double decode(uint16_t bits, int fmt)
{
    return fmt == 0 ? oracle_f16_to_f64(bits) : oracle_bf16_to_f64(bits);
}

/* Decode a whole array (used by the tests to pin the decoders exhaustively). */
void oracle_decode(const uint16_t *src, double *dst, int64_t n, int fmt)
{
    for (int64_t t = 0; t < n; ++t) dst[t] = decode(src[t], fmt);
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_num_procs();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void)
{
    return set_threads(0);
}

/*
 * C[i][j] = sum_k A[i][k] * B[j][k] in fp64 for fp16 (fmt 0) or bf16 (fmt 1) operands.
 * Returns 0 on success, -1 on a bad argument or allocation failure.
 * Rows of C are independent, so rows are spread over `nthreads` OpenMP threads
 * (<= 0: all processors); each element is still one sequential sum over k.
 */
int oracle_gemm_tn_half(const uint16_t *A, const uint16_t *B, double *C,
                        int64_t M, int64_t N, int64_t K, int fmt, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (fmt != 0 && fmt != 1)) return -1;
    if (M == 0 || N == 0) return 0;
    double *Ad = (double *)malloc(sizeof(double) * (size_t)(M * K + 1));
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(N * K + 1));
    if (!Ad || !Bd) { free(Ad); free(Bd); return -1; }
    for (int64_t t = 0; t < M * K; ++t) Ad[t] = decode(A[t], fmt);
    for (int64_t t = 0; t < N * K; ++t) Bd[t] = decode(B[t], fmt);
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += Ad[i * K + k] * Bd[j * K + k];
            C[i * N + j] = s;
        }
    }
    free(Ad);
    free(Bd);
    return 0;
}

/* The same sum, only at the listed output positions: out[t] = C[rows[t]][cols[t]]. */
int oracle_gemm_tn_half_sampled(const uint16_t *A, const uint16_t *B,
                                int64_t M, int64_t N, int64_t K, int fmt,
                                const int64_t *rows, const int64_t *cols, int64_t n,
                                double *out, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || n < 0 || (fmt != 0 && fmt != 1)) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t *a = A + rows[t] * K;
        const uint16_t *b = B + cols[t] * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += decode(a[k], fmt) * decode(b[k], fmt);
        out[t] = s;
    }
    return 0;
}

/* Two's-complement reduction of an exact integer sum to int32 (wrap modulo 2^32). */
static int32_t wrap_i32(int64_t s)
{
    const uint32_t low = (uint32_t)((uint64_t)s & 0xffffffffu);
    return low >= 0x80000000u ? (int32_t)((int64_t)low - 4294967296LL) : (int32_t)low;
}

/*
 * Exact int8 GEMM: C64[i][j] = sum_k int64(A[i][k]) * int64(B[j][k]); C32 = wrap(C64).
 * Either output pointer may be NULL.
 */
int oracle_gemm_tn_i8(const int8_t *A, const int8_t *B, int64_t *C64, int32_t *C32,
                      int64_t M, int64_t N, int64_t K, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)A[i * K + k] * (int64_t)B[j * K + k];
            if (C64) C64[i * N + j] = s;
            if (C32) C32[i * N + j] = wrap_i32(s);
        }
    }
    return 0;
}

int oracle_gemm_tn_i8_sampled(const int8_t *A, const int8_t *B, int64_t M, int64_t N, int64_t K,
                              const int64_t *rows, const int64_t *cols, int64_t n,
                              int64_t *out64, int32_t *out32, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        const int8_t *a = A + rows[t] * K;
        const int8_t *b = B + cols[t] * K;
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k) s += (int64_t)a[k] * (int64_t)b[k];
        if (out64) out64[t] = s;
        if (out32) out32[t] = wrap_i32(s);
    }
    return 0;
}

/*
 * Fused epilogue of a linear layer: C[i][j] = act(C[i][j] + bias[j]) in fp64, applied to
 * the GEMM result above (bias: N values, may be NULL).  act: 0 none, 1 ReLU max(x, 0),
 * 2 GELU x * Phi(x) with Phi the standard normal CDF = (1 + erf(x / sqrt 2)) / 2,
 * 3 SiLU x / (1 + exp(-x)).  The GEMM post on RL-driven tuning counts the order of fused
 * operations among its tuning dimensions (paragraph on tile size and fusion order) without
 * naming the operations; these are the ones that follow FFN-shaped GEMMs.
 */
static double apply_act(double x, int act)
{
    switch (act) {
        case 1: return x > 0.0 ? x : 0.0;
        case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
        case 3: return x / (1.0 + exp(-x));
        default: return x;
    }
}

int oracle_epilogue(double *C, int64_t M, int64_t N, const float *bias, int act)
{
    if (M < 0 || N < 0 || act < 0 || act > 3) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            const double x = C[i * N + j] + (bias ? (double)bias[j] : 0.0);
            C[i * N + j] = apply_act(x, act);
        }
    return 0;
}

/* The same at sampled positions: out[t] = act(C[rows[t]][cols[t]] + bias[cols[t]]). */
int oracle_epilogue_sampled(double *vals, const int64_t *cols, int64_t n, const float *bias, int act)
{
    if (n < 0 || act < 0 || act > 3) return -1;
    for (int64_t t = 0; t < n; ++t)
        vals[t] = apply_act(vals[t] + (bias ? (double)bias[cols[t]] : 0.0), act);
    return 0;
}

/*
 * TMA intensity experiment ("B-08. Hopper TMA：从单线程 Bulk Copy 到吞吐墙", sections 5 and
 * 5.2): every element x of the input passes through `iters` fused multiply-adds,
 * y <- fma(y, a, b) starting from y = x, and lands at the same index of the output.  The
 * page fixes the workload (4 KiB tiles, a sweep over the FMA count) but not the arithmetic
 * constants; a and b are arguments.  fmaf is the single-rounding fp32 fused multiply-add of
 * C99, so the result is bit-defined.
 */
int oracle_fma_chain(const float *in, float *out, int64_t n, int iters, float a, float b)
{
    if (n < 0 || iters < 0) return -1;
    for (int64_t t = 0; t < n; ++t) {
        float y = in[t];
        for (int i = 0; i < iters; ++i) y = fmaf(y, a, b);
        out[t] = y;
    }
    return 0;
}
