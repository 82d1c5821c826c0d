// gemm_probe.cu -- gemm_probe_mma_rate: back-to-back tcgen05.mma issue rate per SM
// (declared in include/gemm_probe.h).
//
// One thread per CTA issues `iters` M=128 N=256 K=16 f16 MMAs into one TMEM
// accumulator from zeroed shared-memory operands (the same instruction,
// descriptors and K steps as the GEMM's main loop, without the copies that
// feed it), commits them to an mbarrier and waits with a %globaltimer bound.
// The interval from the first issue to the barrier's completion, in SM cycles,
// gives the dense FLOP per clock of one SM.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "gemm_probe.h"

namespace gbg {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeN = 256;
constexpr uint32_t kProbeATile = kBM * kBK * 2;        // 16 KiB
constexpr uint32_t kProbeBTile = kProbeN * kBK * 2;    // 32 KiB
// More than half of an SM's shared memory, so at most one CTA runs per SM.
constexpr size_t kProbeSmem = 120 * 1024;
constexpr uint64_t kProbeTimeoutNs = 2000000000ull;

__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_rate_kernel(int32_t iters, long long* cycles, long long* ns, int32_t* error_word) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ alignas(8) uint64_t done_bar;
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int warp = static_cast<int>(threadIdx.x) / 32;

    // Zero operands: the rate does not depend on the values, and zeros keep the
    // accumulator finite.
    uint4* z = reinterpret_cast<uint4*>(smem);
    for (uint32_t i = threadIdx.x; i < (kProbeATile + kProbeBTile) / 16; i += kProbeThreads)
        z[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();   // generic-proxy writes, read by the tensor core
    if (warp == 0) {
        tmem_alloc(smem_addr(&tmem_slot), kProbeN);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        mbar_init(smem_addr(&done_bar), 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 1 && elect_one_sync()) {
        const uint32_t a0 = smem_addr(smem);
        const uint64_t a_desc = sw128_kmajor_desc(a0);
        const uint64_t b_desc = sw128_kmajor_desc(a0 + kProbeATile);
        const uint32_t idesc = (1u << 4)                                  // D fp32, A/B fp16, K-major
                               | (static_cast<uint32_t>(kProbeN >> 3) << 17)
                               | (static_cast<uint32_t>(kBM >> 4) << 24);
        const long long c0 = clock64();
        const uint64_t g0 = global_timer_ns();
        for (int32_t i = 0; i < iters; ++i) {
            const uint32_t k = static_cast<uint32_t>(i & 3);   // the four K=16 steps of a k-block
            umma_f16(tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, i > 0 ? 1u : 0u);
        }
        umma_commit(smem_addr(&done_bar));
        bool ok = true;
        while (!mbar_try_wait(smem_addr(&done_bar), 0)) {
            if (global_timer_ns() - g0 > kProbeTimeoutNs) {
                ok = false;
                break;
            }
        }
        const long long c1 = clock64();
        const uint64_t g1 = global_timer_ns();
        if (ok) {
            cycles[blockIdx.x] = c1 - c0;
            ns[blockIdx.x] = static_cast<long long>(g1 - g0);
        } else {
            cycles[blockIdx.x] = -1;
            ns[blockIdx.x] = -1;
            atomicExch(error_word, 1);
            // let the issued MMAs finish before TMEM is released (bounded)
            wait_phase_unwind(smem_addr(&done_bar), 0, 100000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kProbeN);
    }
}

}  // namespace
}  // namespace gbg

extern "C" gemm_status_t gemm_probe_mma_rate(int32_t grid, int32_t iters, int64_t* cycles,
                                             int64_t* ns, int32_t* error_word, void* stream) {
    if (grid < 1 || iters < 1 || iters > (1 << 24) || !cycles || !ns || !error_word)
        return GEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (grid > sms) return GEMM_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(gbg::mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(gbg::kProbeSmem)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    gbg::mma_rate_kernel<<<grid, gbg::kProbeThreads, gbg::kProbeSmem,
                           reinterpret_cast<cudaStream_t>(stream)>>>(
        iters, reinterpret_cast<long long*>(cycles), reinterpret_cast<long long*>(ns), error_word);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}
