// tma_intensity.cu -- the tutorial page's load-mode x compute-intensity
// experiment, run on GB300 ("B-08. Hopper TMA：从单线程 Bulk Copy 到吞吐墙",
// sections 3 and 5): how much a TMA copy helps depends on whether it overlaps
// compute.  Every element x of `in` becomes y = fma(...fma(x, a, b)..., a, b)
// (fma_iters times) at the same index of `out`; only the way each 4 KiB tile
// reaches shared memory differs:
//   0 sync     : all 256 threads load the tile with plain loads, then compute;
//   1 bulk1d   : one elected thread issues a 1-D cp.async.bulk of the tile and
//                everybody waits on its mbarrier at once (no overlap);
//   2 tensor2d : as bulk1d with a 2-D tensor map and a 32 x 32 tile;
//   3 pipe2    : 1-D bulk copies double-buffered: tile t+1 is in flight while
//                tile t is computed.
// Workload of the page: 64 tiles per 256-thread block, 1-D tiles = 1024
// consecutive floats, 2-D tiles = 32 x 32 squares of a rows x cols matrix.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "tma_intensity.h"

namespace {

constexpr int kTile = 1024;         // floats per tile (4 KiB)
constexpr int kTilesPerBlock = 64;
constexpr int kThreadsPerBlock = 256;
constexpr int kSide = 32;           // 2-D tile edge
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void bar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; on expiry records code 1 in the error word (if any) and returns false.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, int32_t* err) {
    if (bar_test(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!bar_test(bar, parity)) {
        if (now_ns() - t0 > kWaitLimitNs) {
            if (err) atomicCAS(err, 0, 1);
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tensor_g2s(uint32_t dst, const CUtensorMap* map, int32_t x,
                                           int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ float fma_chain(float y, int iters, float a, float b) {
    for (int i = 0; i < iters; ++i) y = fmaf(y, a, b);
    return y;
}

template <int MODE>
__global__ void __launch_bounds__(kThreadsPerBlock)
    tma_intensity_kernel(const __grid_constant__ CUtensorMap tmap, const float* __restrict__ in,
                         float* __restrict__ out, int32_t cols, int iters, float a, float b,
                         int32_t* err) {
    __shared__ __align__(1024) float tile[2][kTile];
    __shared__ __align__(8) uint64_t bar[2];
    const int tid = static_cast<int>(threadIdx.x);
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kTilesPerBlock;
    if (MODE != 0 && tid == 0) {
        bar_init(saddr(&bar[0]));
        bar_init(saddr(&bar[1]));
    }
    __syncthreads();

    if constexpr (MODE == 0) {
        for (int t = 0; t < kTilesPerBlock; ++t) {
            const int64_t base = (first + t) * kTile;
#pragma unroll
            for (int e = 0; e < kTile / kThreadsPerBlock; ++e)
                tile[0][tid + e * kThreadsPerBlock] = in[base + tid + e * kThreadsPerBlock];
            __syncthreads();
#pragma unroll
            for (int e = 0; e < kTile / kThreadsPerBlock; ++e)
                out[base + tid + e * kThreadsPerBlock] =
                    fma_chain(tile[0][tid + e * kThreadsPerBlock], iters, a, b);
            __syncthreads();
        }
    } else if constexpr (MODE == 1 || MODE == 2) {
        const int tiles_x = cols / kSide;
        uint32_t phase = 0;
        for (int t = 0; t < kTilesPerBlock; ++t) {
            const int64_t g = first + t;
            if (tid == 0) {
                bar_expect(saddr(&bar[0]), kTile * 4);
                if constexpr (MODE == 1)
                    bulk_g2s(saddr(tile[0]), in + g * kTile, kTile * 4, saddr(&bar[0]));
                else
                    tensor_g2s(saddr(tile[0]), &tmap, static_cast<int32_t>(g % tiles_x) * kSide,
                               static_cast<int32_t>(g / tiles_x) * kSide, saddr(&bar[0]));
            }
            bar_wait(saddr(&bar[0]), phase, err);   // immediate wait: no overlap
            phase ^= 1u;
#pragma unroll
            for (int e = 0; e < kTile / kThreadsPerBlock; ++e) {
                const int idx = tid + e * kThreadsPerBlock;
                const float y = fma_chain(tile[0][idx], iters, a, b);
                if constexpr (MODE == 1) {
                    out[g * kTile + idx] = y;
                } else {
                    const int64_t row = (g / tiles_x) * kSide + idx / kSide;
                    const int64_t col = (g % tiles_x) * kSide + idx % kSide;
                    out[row * cols + col] = y;
                }
            }
            __syncthreads();   // the tile buffer is refilled next iteration
        }
    } else {
        // pipe2: tile t+1 in flight while tile t is computed.
        if (tid == 0) {
            bar_expect(saddr(&bar[0]), kTile * 4);
            bulk_g2s(saddr(tile[0]), in + first * kTile, kTile * 4, saddr(&bar[0]));
        }
        for (int t = 0; t < kTilesPerBlock; ++t) {
            const int buf = t & 1;
            if (tid == 0 && t + 1 < kTilesPerBlock) {
                // the other buffer was released by the __syncthreads ending tile t-1
                bar_expect(saddr(&bar[buf ^ 1]), kTile * 4);
                bulk_g2s(saddr(tile[buf ^ 1]), in + (first + t + 1) * kTile, kTile * 4,
                         saddr(&bar[buf ^ 1]));
            }
            bar_wait(saddr(&bar[buf]), static_cast<uint32_t>((t >> 1) & 1), err);
            const int64_t base = (first + t) * kTile;
#pragma unroll
            for (int e = 0; e < kTile / kThreadsPerBlock; ++e)
                out[base + tid + e * kThreadsPerBlock] =
                    fma_chain(tile[buf][tid + e * kThreadsPerBlock], iters, a, b);
            __syncthreads();
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

extern "C" gemm_status_t tma_intensity_run(int32_t mode, int32_t fma_iters, float a, float b,
                                           const float* in, float* out, int64_t n, int32_t cols,
                                           int32_t* error_word, void* stream_ptr) {
    if (mode < 0 || mode > 3 || fma_iters < 0 || n <= 0 || !in || !out) return GEMM_ERR_INVALID_ARG;
    const int64_t per_block = static_cast<int64_t>(kTile) * kTilesPerBlock;
    if (n % per_block != 0 || n / per_block > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u)
        return GEMM_ERR_ALIGNMENT;
    CUtensorMap map = {};
    if (mode == 2) {
        if (cols <= 0 || cols % kSide != 0 || n % cols != 0 || (n / cols) % kSide != 0)
            return GEMM_ERR_INVALID_ARG;
        PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
        if (!fn) return GEMM_ERR_TENSORMAP;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(n / cols)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
        const cuuint32_t box[2] = {kSide, kSide};
        const cuuint32_t estr[2] = {1, 1};
        if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(in), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GEMM_ERR_TENSORMAP;
    }
    const unsigned grid = static_cast<unsigned>(n / per_block);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_ptr);
    switch (mode) {
        case 0: tma_intensity_kernel<0><<<grid, kThreadsPerBlock, 0, s>>>(map, in, out, cols, fma_iters, a, b, error_word); break;
        case 1: tma_intensity_kernel<1><<<grid, kThreadsPerBlock, 0, s>>>(map, in, out, cols, fma_iters, a, b, error_word); break;
        case 2: tma_intensity_kernel<2><<<grid, kThreadsPerBlock, 0, s>>>(map, in, out, cols, fma_iters, a, b, error_word); break;
        default: tma_intensity_kernel<3><<<grid, kThreadsPerBlock, 0, s>>>(map, in, out, cols, fma_iters, a, b, error_word); break;
    }
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}
