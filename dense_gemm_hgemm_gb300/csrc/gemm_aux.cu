// gemm_aux.cu -- small HBM-bound kernels around the GEMM:
//   * widen_i8: int8 operands -> fp16 copies (every int8 value is exact in fp16),
//     the input side of the integer mode of the tensor-core kernel;
//   * zero_fill: C = 0 for K == 0 (the empty sum); fill_bias_act: C = act(bias)
//     for K == 0 with a bias;
//   * empty: a kernel with no body, for measuring the launch-latency floor.
// The widening and fill kernels are grid-stride loops over 16-byte vectors,
// launched with at most eight 256-thread blocks per SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gemm_launch.h"

namespace gbg {
namespace {

// Four int8 values (one 32-bit word, element 0 in the low byte) -> four fp16
// values (two 32-bit words, element 0 in the low half), exactly.  With
// u = x + 128 in [0, 255] (the byte with its top bit flipped), the fp16 bit
// pattern 0x64 followed by the byte u is 1024 + u: exponent 10, and u fills the
// low eight of the ten fraction bits, one unit in the last place apart.
// Subtracting 1152 = 1024 + 128 (0x6480) leaves x; both operands and the
// difference are integers of at most 11 significant bits, so nothing rounds.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t l = __byte_perm(u, 0x64646464u, 0x5140);   // u0 | 0x64 << 8 | u1 << 16 | 0x64 << 24
    const uint32_t h = __byte_perm(u, 0x64646464u, 0x7362);   // u2, 0x64, u3, 0x64
    const __half2 off = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6480u)));
    const __half2 rl = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
    const __half2 rh = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
    lo = *reinterpret_cast<const uint32_t*>(&rl);
    hi = *reinterpret_cast<const uint32_t*>(&rh);
}

__device__ __forceinline__ void widen16(const uint4& v, uint4& lo, uint4& hi) {
    widen4(v.x, lo.x, lo.y);
    widen4(v.y, lo.z, lo.w);
    widen4(v.z, hi.x, hi.y);
    widen4(v.w, hi.z, hi.w);
}

// na, nb: number of 16-element groups of A and of B.  Each thread has four
// independent 16-byte loads in flight before it converts and stores.
__global__ void __launch_bounds__(256) widen_i8_kernel(const uint4* __restrict__ a, int64_t na,
                                                       const uint4* __restrict__ b, int64_t nb,
                                                       uint4* __restrict__ a16,
                                                       uint4* __restrict__ b16) {
    constexpr int kU = 4;
    const int64_t total = na + nb;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    auto src = [&](int64_t e) { return e < na ? a + e : b + (e - na); };
    auto dst = [&](int64_t e) { return e < na ? a16 + 2 * e : b16 + 2 * (e - na); };
    for (; g + (kU - 1) * stride < total; g += kU * stride) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) v[u] = __ldg(src(g + u * stride));
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            uint4 lo, hi;
            widen16(v[u], lo, hi);
            uint4* d = dst(g + u * stride);
            d[0] = lo;
            d[1] = hi;
        }
    }
    for (; g < total; g += stride) {
        uint4 lo, hi;
        widen16(__ldg(src(g)), lo, hi);
        uint4* d = dst(g);
        d[0] = lo;
        d[1] = hi;
    }
}

// Same launch shape and programmatic-dependent-launch protocol as the GEMM
// kernels, no work: back-to-back launches measure the floor a GEMM launch
// chain can reach.
__global__ void __launch_bounds__(192) empty_kernel() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__global__ void __launch_bounds__(256) zero_fill_kernel(uint4* __restrict__ dst, int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = make_uint4(0u, 0u, 0u, 0u);
}

// K == 0 with a bias: every row of C is act(bias) (the empty sum is 0).
__device__ __forceinline__ float act_of(float x, int act) {
    switch (act) {
        case 1: return fmaxf(x, 0.0f);
        case 2: return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
        case 3: return x / (1.0f + expf(-x));
        default: return x;
    }
}

__global__ void __launch_bounds__(256) fill_bias_act_kernel(void* __restrict__ C, int64_t M,
                                                            int64_t N, const float* __restrict__ bias,
                                                            int act, int bf16) {
    const int64_t total = M * N;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const float v = act_of(bias[i % N], act);
        if (bf16)
            reinterpret_cast<__nv_bfloat16*>(C)[i] = __float2bfloat16_rn(v);
        else
            reinterpret_cast<__half*>(C)[i] = __float2half_rn(v);
    }
}

int grid_for(int64_t work_items, int num_sms) {
    const int64_t per_wave = static_cast<int64_t>(num_sms) * 8;    // 8 x 256 threads per SM
    int64_t blocks = (work_items + 255) / 256;
    if (blocks > per_wave) blocks = per_wave;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_widen_i8(const int8_t* a, int64_t na, const int8_t* b, int64_t nb, void* a16,
                            void* b16, int num_sms, cudaStream_t stream) {
    // na, nb are element counts, multiples of 16 (K % 16 == 0).
    const int64_t ga = na / 16, gb = nb / 16;
    widen_i8_kernel<<<grid_for(ga + gb, num_sms), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(a), ga, reinterpret_cast<const uint4*>(b), gb,
        reinterpret_cast<uint4*>(a16), reinterpret_cast<uint4*>(b16));
    return cudaGetLastError();
}

cudaError_t launch_empty(int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, empty_kernel);
}

cudaError_t launch_fill_bias_act(void* C, int64_t M, int64_t N, const float* bias, int act,
                                 int bf16, int num_sms, cudaStream_t stream) {
    fill_bias_act_kernel<<<grid_for(M * N, num_sms), 256, 0, stream>>>(C, M, N, bias, act, bf16);
    return cudaGetLastError();
}

cudaError_t launch_zero_fill(void* dst, int64_t bytes, int num_sms, cudaStream_t stream) {
    const int64_t n = bytes / 16;   // C rows are multiples of 16 bytes
    zero_fill_kernel<<<grid_for(n, num_sms), 256, 0, stream>>>(reinterpret_cast<uint4*>(dst), n);
    return cudaGetLastError();
}

}  // namespace gbg
