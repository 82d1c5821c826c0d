// gemm_noalloc.cu -- gemm_run_splitk_noalloc: the split-K GEMM with no device
// allocation at all.
//
// Who needs it: callers that may not allocate device memory when they run a
// GEMM -- plugins whose host framework owns all device memory and hands out no
// allocator, services that reserve their memory budget at start-up and forbid
// allocation afterwards, and latency-critical loops where cudaMalloc (which
// can synchronise the device and can fail under fragmentation) is not
// acceptable.  The plan API allocates its split-K scratch in gemm_plan_create;
// this entry point instead uses one fixed scratch array compiled into the
// library (g_noalloc_scratch below).
//
// The array is a file-scope __device__ variable: every GPU on which this
// file's device code is loaded holds its 16 MiB until the process exits (with
// CUDA's lazy module loading, from the first call on that device).  Host code
// cannot use the symbol itself as a device address, so the first call on each
// device (with that device current) asks the runtime for the address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls share the array and it keeps the last call's contents:
// each call clears the split-K counters on its stream before the kernel runs
// (the partials are fully written before they are read), and calls whose
// kernels overlap on the GPU race on the array.  The error word is not cleared
// by a call: a wait that ran out stays recorded until gemm_noalloc_check reads
// and clears it, so one check after several calls sees a failure in any of them.
//
// Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "gemm.h"
#include "gemm_kernel.cuh"
#include "gemm_launch.h"

namespace {

constexpr size_t kScratchBytes = size_t{16} << 20;   // 16 MiB
constexpr size_t kErrorOff = 0;                        // int32 error word
constexpr size_t kCountersOff = 256;                   // uint32 per output tile
constexpr int64_t kMaxTiles = 4096;                    // 16 KiB of counters
constexpr size_t kPartialsOff = 32768;                 // fp32 partials [units][128][64]
constexpr size_t kPartialsBytes = kScratchBytes - kPartialsOff;
constexpr int kBlockN = 64;
constexpr int kStages = 8;
constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceSetup {
    std::once_flag once;
    gemm_status_t status = GEMM_ERR_CUDA;
    unsigned char* scratch = nullptr;
    int num_sms = 0;
    std::atomic<int> ready{0};   // 1 once the set-up succeeded (read without the once flag)
};
DeviceSetup g_setup[kMaxDevices];

// Failure-test hook (gemm_noalloc_set_wait_test): extra bytes every ring slot
// waits for, and the wait limit.  Process-wide; 0 = normal operation.
uint32_t g_wait_test_bytes = 0;
uint64_t g_timeout_ns = kTimeoutNs;

template <int OUT>
cudaError_t allow_smem() {
    return cudaFuncSetAttribute(gbg::gemm_tn_kernel<kBlockN, kStages, OUT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(gbg::SmemLayout<kBlockN, kStages>::kTotal));
}

// Runs once per device, with that device current.
void setup_device(int dev, DeviceSetup* s) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        s->status = GEMM_ERR_CUDA;
        return;
    }
    int sms = 0;
    if (allow_smem<gbg::kOutF16>() != cudaSuccess || allow_smem<gbg::kOutBF16>() != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        s->status = GEMM_ERR_CUDA;
        return;
    }
    s->scratch = static_cast<unsigned char*>(ptr);
    s->num_sms = sms;
    s->status = GEMM_OK;
    s->ready.store(1, std::memory_order_release);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_entry() {
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

bool encode_operand(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
                    CUtensorMapDataType dt) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_entry();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gbg::kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_result(CUtensorMap* map, void* base, int64_t M, int64_t N, CUtensorMapDataType dt) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_entry();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
    const cuuint32_t box[2] = {64, 32};   // 128-byte row segments x 32 rows
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" gemm_status_t gemm_run_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                                 gemm_dtype_t dtype, int32_t split_k,
                                                 const void* A, const void* B, void* C,
                                                 void* stream_ptr) {
    if (dtype != GEMM_F16 && dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0 || split_k < 1) return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 15u)
        return GEMM_ERR_ALIGNMENT;

    const int64_t m_blocks = (M + gbg::kBM - 1) / gbg::kBM;
    const int64_t n_blocks = (N + kBlockN - 1) / kBlockN;
    const int64_t tiles = m_blocks * n_blocks;
    const int64_t num_kb = (K + gbg::kBK - 1) / gbg::kBK;
    int64_t s = split_k;
    if (s > num_kb && num_kb > 0) s = num_kb;
    if (num_kb == 0) s = 1;
    const int64_t per = num_kb > 0 ? (num_kb + s - 1) / s : 0;
    if (per > 0) s = (num_kb + per - 1) / per;
    if (tiles * s > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (s > 1 && (tiles > kMaxTiles ||
                  static_cast<size_t>(tiles * s) * gbg::kBM * kBlockN * 4 > kPartialsBytes))
        return GEMM_ERR_SCRATCH_LIMIT;

    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_ARCH;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    DeviceSetup& su = g_setup[dev];
    std::call_once(su.once, setup_device, dev, &su);
    if (su.status != GEMM_OK) return su.status;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    if (K == 0) {
        if (gbg::launch_zero_fill(C, M * N * 2, su.num_sms, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }

    // Split-K counters start at zero for this call (the error word is sticky
    // until gemm_noalloc_check).
    if (cudaMemsetAsync(su.scratch + kCountersOff, 0, kPartialsOff - kCountersOff, stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }

    const CUtensorMapDataType dt =
        dtype == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap map_a, map_b, map_c;
    if (!encode_operand(&map_a, A, M, K, gbg::kBM, dt) ||
        !encode_operand(&map_b, B, N, K, kBlockN, dt) || !encode_result(&map_c, C, M, N, dt))
        return GEMM_ERR_TENSORMAP;

    gbg::KParams kp;
    memset(&kp, 0, sizeof(kp));
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.K = static_cast<int32_t>(K);
    kp.num_kb = static_cast<int32_t>(num_kb);
    kp.m_blocks = static_cast<int32_t>(m_blocks);
    kp.n_blocks = static_cast<int32_t>(n_blocks);
    kp.split_k = static_cast<int32_t>(s);
    kp.kb_per_split = static_cast<int32_t>(per);
    kp.chunk_kb = static_cast<int32_t>(per);
    kp.raster_group = static_cast<int32_t>(m_blocks < 16 ? m_blocks : 16);
    kp.num_units = static_cast<int32_t>(tiles * s);
    gbg::set_divisors(&kp);
    const uint32_t fmt = dtype == GEMM_BF16 ? 1u : 0u;
    kp.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) |
               (static_cast<uint32_t>(kBlockN >> 3) << 17) |
               (static_cast<uint32_t>(gbg::kBM >> 4) << 24);
    kp.tx_extra = g_wait_test_bytes;
    kp.C = C;
    kp.workspace = su.scratch + kPartialsOff;
    kp.counters = reinterpret_cast<uint32_t*>(su.scratch + kCountersOff);
    kp.error_word = reinterpret_cast<int32_t*>(su.scratch + kErrorOff);
    kp.timeout_ns = g_timeout_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kp.num_units < su.num_sms ? kp.num_units : su.num_sms));
    cfg.blockDim = dim3(gbg::kThreads);
    cfg.dynamicSmemBytes = gbg::SmemLayout<kBlockN, kStages>::kTotal;
    cfg.stream = stream;
    const cudaError_t e =
        dtype == GEMM_BF16
            ? cudaLaunchKernelEx(&cfg, gbg::gemm_tn_kernel<kBlockN, kStages, gbg::kOutBF16>, map_a,
                                 map_b, map_c, kp)
            : cudaLaunchKernelEx(&cfg, gbg::gemm_tn_kernel<kBlockN, kStages, gbg::kOutF16>, map_a,
                                 map_b, map_c, kp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

extern "C" gemm_status_t gemm_noalloc_check(void* stream_ptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    DeviceSetup& su = g_setup[dev];
    // No call has run on this device yet (the set-up of the first call is what
    // resolves the array's address): nothing can have failed.
    if (su.ready.load(std::memory_order_acquire) == 0) return GEMM_OK;
    int32_t word = 0;
    if (cudaMemcpy(&word, su.scratch + kErrorOff, sizeof(word), cudaMemcpyDeviceToHost) !=
        cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (word == 0) return GEMM_OK;
    const int32_t zero = 0;
    if (cudaMemcpy(su.scratch + kErrorOff, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_ERR_DEVICE_TIMEOUT;
}

extern "C" gemm_status_t gemm_noalloc_set_wait_test(uint32_t extra_bytes, uint64_t timeout_ns) {
    if (extra_bytes > 4096 || (extra_bytes & 15u)) return GEMM_ERR_INVALID_ARG;
    g_wait_test_bytes = extra_bytes;
    g_timeout_ns = timeout_ns ? timeout_ns : kTimeoutNs;
    return GEMM_OK;
}
