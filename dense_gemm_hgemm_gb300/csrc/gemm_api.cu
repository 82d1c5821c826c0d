// gemm_api.cu -- the C ABI declared in include/gemm.h.
//
// Host-side work only: argument and alignment validation, configuration choice,
// plan memory, tensor-map encoding (cuTensorMapEncodeTiled obtained through
// cudaGetDriverEntryPointByVersion, so the library needs no -lcuda), and the
// launches.  Every GEMM step runs in the kernels of gemm_inst_*.cu and
// gemm_aux.cu; there is no host or library fallback.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>

#include "gemm.h"
#include "gemm_config.h"
#include "gemm_launch.h"
#include "gemm_sched.h"

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct PlanMemory {
    size_t error_off, counters_off, ws_off, a16_off, b16_off, total;
};

}  // namespace

struct gemm_plan {
    int64_t M, N, K;
    gemm_dtype_t dtype;
    gemm_layout_t layout;
    gemm_config_t cfg;          // effective configuration
    int device;
    int num_sms;
    int out_kind;
    int form;                   // the kernel's compiled form (gbg::KernelForm) for the plan
    gbg::LaunchShape shape;
    gbg::KParams kp;
    PlanMemory mem;
    uint8_t* dmem;              // one device allocation holding everything below
    int32_t* d_error;
    uint32_t* d_counters;
    void* d_ws;
    void* d_a16;
    void* d_b16;
    const void* map_a_src;      // tensor-map cache keys
    const void* map_b_src;
    const void* map_c_src;
    bool map_a_valid, map_b_valid, map_c_valid;
    CUtensorMap map_a, map_b, map_c;
    // The GEMM launch, fixed at plan creation (a call sets only the stream): the
    // kernel's driver function handle, grid / block / shared memory, programmatic
    // dependent launch and the cluster shape.
    CUfunction fn;
    CUfunction fn_epilogue;     // for calls with a fused bias or activation: the epilogue
                                // form of a plain plan, else the general form
    CUlaunchConfig launch;
    CUlaunchAttribute launch_attr[2];
};

namespace {

bool a_mn_major(gemm_layout_t l) { return l == GEMM_LAYOUT_TT || l == GEMM_LAYOUT_NT; }
bool b_mn_major(gemm_layout_t l) { return l == GEMM_LAYOUT_NN || l == GEMM_LAYOUT_NT; }

gemm_status_t validate_shape(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                             gemm_layout_t layout) {
    if (dtype != GEMM_F16 && dtype != GEMM_BF16 && dtype != GEMM_I8_I32) return GEMM_ERR_UNSUPPORTED;
    if (layout < GEMM_LAYOUT_TN || layout > GEMM_LAYOUT_NT) return GEMM_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    const bool i8 = dtype == GEMM_I8_I32;
    // Stored rows must be multiples of 16 bytes: the contiguous extent of A
    // (K, or M when A is stored K x M) and of B (K, or N), and N * out_bytes for C.
    const int64_t in_mult = i8 ? 16 : 8;
    if ((a_mn_major(layout) ? M : K) % in_mult != 0) return GEMM_ERR_ALIGNMENT;
    if ((b_mn_major(layout) ? N : K) % in_mult != 0) return GEMM_ERR_ALIGNMENT;
    if (N % (i8 ? 4 : 8) != 0) return GEMM_ERR_ALIGNMENT;
    // Work-decomposition indices are 32-bit.
    const int64_t tiles = ((M + gbg::kBM - 1) / gbg::kBM) * ((N + 63) / 64);
    if (tiles > (int64_t{1} << 30)) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

bool valid_block_n(int bn) { return bn == 64 || bn == 128 || bn == 224 || bn == 256; }

// Fill the derived fields of a configuration for a shape (split-K made exact:
// every K slice non-empty).  Returns GEMM_ERR_INVALID_ARG for a bad config.
gemm_status_t normalise_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                               const gemm_config_t& in, gemm_config_t* out,
                               int32_t* kb_per_split) {
    gemm_config_t c = in;
    if (!valid_block_n(c.block_n)) return GEMM_ERR_INVALID_ARG;
    if (c.cta_pair != 0 && c.cta_pair != 1) return GEMM_ERR_INVALID_ARG;
    if (c.direct_store != 0 && c.direct_store != 1) return GEMM_ERR_INVALID_ARG;
    if (c.direct_store && c.cta_pair) return GEMM_ERR_INVALID_ARG;
    if (c.multicast == 1) c.multicast = 0;   // 0 and 1 both mean off
    if (c.multicast != 0 && c.multicast != 2 && c.multicast != 4) return GEMM_ERR_INVALID_ARG;
    if (c.l2_prefetch < 0 || c.l2_prefetch > 64) return GEMM_ERR_INVALID_ARG;
    if (c.kblocks_per_stage == 0) c.kblocks_per_stage = 1;
    if (c.kblocks_per_stage != 1 && c.kblocks_per_stage != 2 && c.kblocks_per_stage != 4)
        return GEMM_ERR_INVALID_ARG;
    if (c.kblocks_per_stage > 1 && c.multicast > 1) return GEMM_ERR_INVALID_ARG;
    if (c.kblocks_per_stage == 2 && !c.cta_pair && c.block_n > 128) return GEMM_ERR_INVALID_ARG;
    // four k-blocks per slot: two 96 KiB slots, one-SM 64-wide or SM-pair 128-wide tiles
    if (c.kblocks_per_stage == 4 && c.block_n != (c.cta_pair ? 128 : 64))
        return GEMM_ERR_INVALID_ARG;
    // 224-wide tiles: SM pairs only, one K slice, no multicast (each CTA's 112 B
    // rows are one copy box; the epilogue stores the last 32 columns directly)
    if (c.block_n == 224 && (!c.cta_pair || c.split_k != 1 || c.multicast > 1))
        return GEMM_ERR_INVALID_ARG;
    // Integer tiles keep their int32 sums in registers: up to 128 columns on one SM,
    // 224/256 on SM pairs with eight epilogue warps (one K slice, no multicast).
    if (dtype == GEMM_I8_I32 && c.block_n > 128 &&
        (!c.cta_pair || c.split_k != 1 || c.multicast > 1))
        return GEMM_ERR_INVALID_ARG;
    if (c.cta_pair) {
        // SM pair: 256-row tiles; K is sliced only across the pairs of a cluster.
        if (c.block_n < 128) return GEMM_ERR_INVALID_ARG;
        if (c.split_k != 1 && c.split_mode != 1) return GEMM_ERR_INVALID_ARG;
    }
    const int want_stages = gbg::default_ring_stages(c.cta_pair, c.block_n, c.kblocks_per_stage);
    if (c.stages == 0) c.stages = want_stages;
    if (c.stages != want_stages) return GEMM_ERR_INVALID_ARG;
    if (c.split_k < 1 || c.raster_group < 1 || c.max_ctas < 0) return GEMM_ERR_INVALID_ARG;
    if (c.split_mode != 0 && c.split_mode != 1) return GEMM_ERR_INVALID_ARG;
    const int64_t num_kb = (K + gbg::kBK - 1) / gbg::kBK;
    int64_t s = c.split_k;
    if (num_kb == 0) s = 1;
    if (s > num_kb && num_kb > 0) s = num_kb;
    const int64_t per = num_kb > 0 ? (num_kb + s - 1) / s : 0;
    if (per > 0) s = (num_kb + per - 1) / per;
    const int64_t tile_m = c.cta_pair ? 2 * gbg::kBM : gbg::kBM;
    const int64_t m_blocks = (M + tile_m - 1) / tile_m;
    const int64_t n_blocks = (N + c.block_n - 1) / c.block_n;
    if (m_blocks * n_blocks * s > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    c.split_k = static_cast<int32_t>(s);
    if (c.split_k == 1) c.split_mode = 0;
    if (c.multicast > 1 && c.split_k != 1) return GEMM_ERR_INVALID_ARG;
    // SM pairs share A between two pairs of one four-CTA cluster
    if (c.multicast > 2 && c.cta_pair) return GEMM_ERR_INVALID_ARG;
    // Cluster split: the slices of a tile share its 128 rows evenly (S | 128) and
    // form a portable cluster (S <= 8).
    if (c.split_mode == 1 && c.split_k != 2 && c.split_k != 4 && c.split_k != 8)
        return GEMM_ERR_INVALID_ARG;
    // ... and with SM pairs the cluster holds 2 * split_k CTAs
    if (c.split_mode == 1 && c.cta_pair && c.split_k > 4) return GEMM_ERR_INVALID_ARG;
    if (c.raster_group > m_blocks && m_blocks > 0) c.raster_group = static_cast<int32_t>(m_blocks);
    *out = c;
    *kb_per_split = static_cast<int32_t>(per);
    return GEMM_OK;
}

PlanMemory plan_memory(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, const gemm_config_t& c) {
    PlanMemory m{};
    size_t off = 0;
    m.error_off = off;
    off += kAlign;
    const int64_t tiles = ((M + gbg::kBM - 1) / gbg::kBM) * ((N + c.block_n - 1) / c.block_n);
    const bool workspace = c.split_k > 1 && c.split_mode == 0;
    m.counters_off = off;
    if (workspace) off += round_up(static_cast<size_t>(tiles) * 4, kAlign);
    m.ws_off = off;
    if (workspace)
        off += round_up(static_cast<size_t>(tiles) * c.split_k * gbg::kBM * c.block_n * 4, kAlign);
    m.a16_off = off;
    if (dtype == GEMM_I8_I32) off += round_up(static_cast<size_t>(M) * K * 2, kAlign);
    m.b16_off = off;
    if (dtype == GEMM_I8_I32) off += round_up(static_cast<size_t>(N) * K * 2, kAlign);
    m.total = off;
    return m;
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

// cuLaunchKernelEx, also through the runtime's driver entry point: a launch with a
// function handle and a prepared configuration costs ~0.12 us less host time per
// call than cudaLaunchKernelEx with the kernel's host stub (measured on GB300 with
// this kernel's 584 bytes of parameters: 1.39 vs 1.51 us).
PFN_cuLaunchKernelEx_v11060 launch_fn() {
    static PFN_cuLaunchKernelEx_v11060 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuLaunchKernelEx", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuLaunchKernelEx_v11060>(p);
    });
    return fn;
}

// 2-D map over a rows x K K-contiguous 16-bit matrix; box = 64 (K) x box_rows,
// 128-byte swizzle (one 64-element row of the box = one 128-byte swizzle span),
// zero fill outside the matrix.
gemm_status_t encode_kmajor(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                            int box_rows, CUtensorMapDataType dt) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return GEMM_ERR_TENSORMAP;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gbg::kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_TENSORMAP;
}

// 2-D map over the M x N row-major C for the epilogue's TMA stores: box = one
// 128-byte row segment (64 16-bit or 32 32-bit values) x 32 rows, 128-byte
// swizzle (the layout the epilogue writes its store buffers in).
gemm_status_t encode_output(CUtensorMap* map, void* base, int64_t M, int64_t N, gemm_dtype_t dt) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return GEMM_ERR_TENSORMAP;
    const int esize = dt == GEMM_I8_I32 ? 4 : 2;
    const CUtensorMapDataType t = dt == GEMM_I8_I32 ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                  : dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * esize};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, t, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_TENSORMAP;
}

// Map over an operand stored K x rows (rows contiguous): boxes of 64 rows-elements
// (128 bytes) x 64 K-rows with 128-byte swizzle, the M/N-major tile blocks the
// kernels' descriptors expect.
gemm_status_t encode_mnmajor(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                             CUtensorMapDataType dt, int kblocks = 1) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return GEMM_ERR_TENSORMAP;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(rows) * 2};
    // kblocks consecutive 64-row K blocks per box (two-k-block ring slots)
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(gbg::kBK * kblocks)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_TENSORMAP;
}

// 3-D view of a K-contiguous rows x K operand (K % 64 == 0) as (64 elements,
// rows, K/64 k-blocks) with strides (K*2 bytes, 128 bytes): one box of
// 64 x box_rows x kblocks brings kblocks consecutive k-blocks of box_rows rows,
// k-block-major in shared memory, 128-byte swizzled like the 2-D boxes.
gemm_status_t encode_kmajor3d(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                              int box_rows, int kblocks, CUtensorMapDataType dt) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return GEMM_ERR_TENSORMAP;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(gbg::kBK), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(K / gbg::kBK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(gbg::kBK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(gbg::kBK), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(kblocks)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_TENSORMAP;
}

// Map for operand A (rows = M) or B (rows = N) in the plan's storage; kblocks = 2
// selects the two-k-block boxes (3-D view of a K-contiguous operand, or 128-row
// boxes of an M/N-contiguous one).
gemm_status_t encode_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K,
                                 int box_rows, bool mn_major, CUtensorMapDataType dt,
                                 int kblocks = 1) {
    if (mn_major) return encode_mnmajor(map, base, rows, K, dt, kblocks);
    if (kblocks > 1) return encode_kmajor3d(map, base, rows, K, box_rows, kblocks, dt);
    return encode_kmajor(map, base, rows, K, box_rows, dt);
}

CUtensorMapDataType operand_type(gemm_dtype_t dt) {
    return dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

gemm_status_t device_of_caller(int* device, int* num_sms) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_ARCH;
    *device = dev;
    *num_sms = sms;
    return GEMM_OK;
}

gemm_status_t create_plan(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                          gemm_layout_t layout, const gemm_config_t* user_cfg, gemm_plan_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    gemm_status_t st = validate_shape(M, N, K, dtype, layout);
    if (st != GEMM_OK) return st;
    // A stored K x M is copied in 64-column blocks: at most two multicast slices
    if (user_cfg && user_cfg->multicast > 2 && a_mn_major(layout)) return GEMM_ERR_INVALID_ARG;
    // ... and so is a B stored K x N: a 224-wide pair tile's 112 rows per CTA are not
    if (user_cfg && user_cfg->block_n == 224 && b_mn_major(layout)) return GEMM_ERR_INVALID_ARG;
    // several k-blocks per slot of a K-contiguous operand come from its 3-D view,
    // which needs K % 64 == 0
    const bool some_k_major = !a_mn_major(layout) || !b_mn_major(layout);
    if (user_cfg && user_cfg->kblocks_per_stage > 1 && some_k_major && K % gbg::kBK != 0)
        return GEMM_ERR_INVALID_ARG;
    if (user_cfg) {
        gemm_config_t tmp;
        int32_t per;
        st = normalise_config(M, N, K, dtype, *user_cfg, &tmp, &per);
        if (st != GEMM_OK) return st;
    }
    int dev = 0, sms = 0;
    st = device_of_caller(&dev, &sms);
    if (st != GEMM_OK) return st;

    gemm_config_t want = user_cfg ? *user_cfg : gbg::select_config(M, N, K, dtype, sms);
    if (want.multicast > 2 && a_mn_major(layout)) want.multicast = 2;
    if (want.block_n == 224 && b_mn_major(layout)) {
        want.block_n = 256;
        want.stages = 0;
    }
    if (want.kblocks_per_stage > 1 && some_k_major && K % gbg::kBK != 0) {
        want.kblocks_per_stage = 1;
        want.stages = 0;
    }
    gemm_config_t cfg;
    int32_t kb_per_split = 0;
    st = normalise_config(M, N, K, dtype, want, &cfg, &kb_per_split);
    if (st != GEMM_OK) return st;

    gemm_plan* p = new (std::nothrow) gemm_plan();
    if (!p) return GEMM_ERR_OOM;
    p->M = M;
    p->N = N;
    p->K = K;
    p->dtype = dtype;
    p->layout = layout;
    p->cfg = cfg;
    p->device = dev;
    p->num_sms = sms;
    p->out_kind = dtype == GEMM_F16 ? gbg::kOutF16 : (dtype == GEMM_BF16 ? gbg::kOutBF16 : gbg::kOutI32);
    p->mem = plan_memory(M, N, K, dtype, cfg);
    if (cudaMalloc(reinterpret_cast<void**>(&p->dmem), p->mem.total) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return GEMM_ERR_OOM;
    }
    if (cudaMemset(p->dmem, 0, p->mem.a16_off) != cudaSuccess) {   // error word + counters
        cudaGetLastError();
        cudaFree(p->dmem);
        delete p;
        return GEMM_ERR_CUDA;
    }
    p->d_error = reinterpret_cast<int32_t*>(p->dmem + p->mem.error_off);
    p->d_counters = reinterpret_cast<uint32_t*>(p->dmem + p->mem.counters_off);
    p->d_ws = p->dmem + p->mem.ws_off;
    p->d_a16 = p->dmem + p->mem.a16_off;
    p->d_b16 = p->dmem + p->mem.b16_off;

    // The kernel's compiled form: plain (or, for one-SM K slices in a cluster,
    // cluster split) when the plan uses none of the modes that form fixes
    // (multicast, per-thread stores, M/N-contiguous operands, an L2 prefetch
    // distance, four k-blocks per slot); its launches reach their copies and
    // stores sooner.  The one-SM integer mode and 128-wide integer SM-pair tiles
    // have the general form only.
    {
        const bool fixed_ok = cfg.multicast <= 1 && !cfg.direct_store && cfg.l2_prefetch == 0 &&
                              !a_mn_major(layout) && !b_mn_major(layout) &&
                              cfg.kblocks_per_stage != 4;
        p->form = gbg::kFormGeneral;
        if (fixed_ok && cfg.cta_pair) {
            if (cfg.split_k == 1 && !(dtype == GEMM_I8_I32 && cfg.block_n == 128))
                p->form = gbg::kFormPlain;
        } else if (fixed_ok && dtype != GEMM_I8_I32) {
            if (cfg.split_k == 1)
                p->form = gbg::kFormPlain;
            else if (cfg.split_mode == 1)
                p->form = gbg::kFormClusterSplit;
        }
    }
    size_t smem = 0;
    const cudaError_t prep =
        gbg::gemm_prepare(cfg.block_n, cfg.stages, p->out_kind, cfg.cta_pair, p->form, &smem);
    if (prep != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->dmem);
        delete p;
        return GEMM_ERR_LAUNCH;
    }

    gbg::KParams& kp = p->kp;
    memset(&kp, 0, sizeof(kp));
    kp.M = static_cast<int32_t>(M);
    kp.N = static_cast<int32_t>(N);
    kp.K = static_cast<int32_t>(K);
    kp.num_kb = static_cast<int32_t>((K + gbg::kBK - 1) / gbg::kBK);
    const int64_t tile_m = cfg.cta_pair ? 2 * gbg::kBM : gbg::kBM;
    kp.m_blocks = static_cast<int32_t>((M + tile_m - 1) / tile_m);
    kp.n_blocks = static_cast<int32_t>((N + cfg.block_n - 1) / cfg.block_n);
    kp.split_k = cfg.split_k;
    kp.cluster_split = cfg.split_mode == 1 ? 1 : 0;
    kp.kb_per_split = kb_per_split;
    // Integer mode: chunks of 16 k-blocks (1024 products of magnitude <= 2^14, so
    // every fp32 partial sum is an integer of magnitude <= 2^24: exactly
    // representable, hence exact).
    kp.chunk_kb = dtype == GEMM_I8_I32 ? 16 : (kb_per_split > 0 ? kb_per_split : 1);
    kp.raster_group = cfg.raster_group;
    kp.direct_store = cfg.direct_store;
    kp.a_mn_major = a_mn_major(layout) ? 1 : 0;
    kp.b_mn_major = b_mn_major(layout) ? 1 : 0;
    kp.mcast = cfg.multicast > 1 ? cfg.multicast : 1;
    kp.l2_prefetch = cfg.l2_prefetch;
    // M <= 64 on one SM: copy only the tile's 64 real A rows (the copy engine would
    // otherwise deliver 64 zero-filled rows at the same cost per byte)
    kp.a_half = (M <= gbg::kBM / 2 && !cfg.cta_pair && kp.mcast == 1) ? 1 : 0;
    // with A multicast a unit is a group of `mcast` adjacent n-blocks
    kp.num_units = kp.mcast > 1 ? kp.m_blocks * ((kp.n_blocks + kp.mcast - 1) / kp.mcast)
                                : kp.m_blocks * kp.n_blocks * kp.split_k;
    gbg::set_divisors(&kp);
    const uint32_t fmt = dtype == GEMM_BF16 ? 1u : 0u;
    kp.idesc = (1u << 4)                                         // D: fp32
               | (fmt << 7) | (fmt << 10)                        // A, B: fp16 or bf16
               | (static_cast<uint32_t>(kp.a_mn_major) << 15)    // A M-major
               | (static_cast<uint32_t>(kp.b_mn_major) << 16)    // B N-major
               | (static_cast<uint32_t>(cfg.block_n >> 3) << 17)  // N / 8
               | (static_cast<uint32_t>(tile_m >> 4) << 24);      // M / 16 (128, or 256 for a pair)
    kp.tx_extra = 0;
    kp.workspace = p->d_ws;
    kp.counters = p->d_counters;
    kp.error_word = p->d_error;
    kp.timeout_ns = kDefaultTimeoutNs;

    const int cap = cfg.max_ctas > 0 ? cfg.max_ctas : sms;
    p->shape.grid = kp.num_units < cap ? kp.num_units : cap;
    p->shape.cluster = 1;
    if (kp.cluster_split) {   // one unit per CTA, clusters of split_k CTAs
        p->shape.grid = kp.num_units;
        p->shape.cluster = cfg.split_k;
    }
    if (kp.mcast > 1) {       // persistent clusters of mcast CTAs per tile group
        const int groups_cap = cap / kp.mcast > 0 ? cap / kp.mcast : 1;
        p->shape.grid = kp.mcast * (kp.num_units < groups_cap ? kp.num_units : groups_cap);
        p->shape.cluster = kp.mcast;
    }
    if (cfg.cta_pair && kp.cluster_split) {   // one unit per pair, split_k pairs per cluster
        p->shape.grid = 2 * kp.num_units;
        p->shape.cluster = 2 * cfg.split_k;
    } else if (cfg.cta_pair && kp.mcast > 1) { // persistent clusters of two pairs sharing A
        const int quads_cap = cap / 4 > 0 ? cap / 4 : 1;
        p->shape.grid = 4 * (kp.num_units < quads_cap ? kp.num_units : quads_cap);
        p->shape.cluster = 4;
    } else if (cfg.cta_pair) {                 // persistent SM pairs: two CTAs per tile
        const int pairs_cap = cap / 2 > 0 ? cap / 2 : 1;
        p->shape.grid = 2 * (kp.num_units < pairs_cap ? kp.num_units : pairs_cap);
        p->shape.cluster = 2;
    }
    if (p->shape.grid < 1) p->shape.grid = 1;
    p->shape.block = cfg.cta_pair ? gbg::pair_threads(cfg.block_n, p->out_kind) : gbg::kThreads;
    p->shape.smem_bytes = smem;
    if (kp.mcast > 1) {   // no more persistent clusters than fit on the GPU at once
        int fit = 0;
        if (gbg::gemm_max_clusters(cfg.block_n, cfg.stages, p->out_kind, cfg.cta_pair, p->form,
                                   p->shape,
                                   &fit) == cudaSuccess && fit > 0) {
            if (p->shape.grid > fit * p->shape.cluster) p->shape.grid = fit * p->shape.cluster;
        } else {
            cudaGetLastError();
        }
    }

    const void* kernel =
        gbg::gemm_kernel_ptr(cfg.block_n, cfg.stages, p->out_kind, cfg.cta_pair, p->form);
    // (integer plans have no fused epilogue: theirs is never launched)
    const int form_epi = p->form == gbg::kFormPlain && dtype != GEMM_I8_I32 ? gbg::kFormEpilogue
                                                                           : gbg::kFormGeneral;
    const void* kernel_epi =
        gbg::gemm_kernel_ptr(cfg.block_n, cfg.stages, p->out_kind, cfg.cta_pair, form_epi);
    size_t smem_epi = 0;
    if (!kernel || !kernel_epi || cudaGetFuncBySymbol(&p->fn, kernel) != cudaSuccess ||
        cudaGetFuncBySymbol(&p->fn_epilogue, kernel_epi) != cudaSuccess || !launch_fn() ||
        (form_epi != p->form &&
         gbg::gemm_prepare(cfg.block_n, cfg.stages, p->out_kind, cfg.cta_pair, form_epi,
                           &smem_epi) != cudaSuccess)) {
        cudaGetLastError();
        cudaFree(p->dmem);
        delete p;
        return GEMM_ERR_LAUNCH;
    }
    memset(&p->launch, 0, sizeof(p->launch));
    p->launch.gridDimX = static_cast<unsigned>(p->shape.grid);
    p->launch.gridDimY = p->launch.gridDimZ = 1;
    p->launch.blockDimX = static_cast<unsigned>(p->shape.block);
    p->launch.blockDimY = p->launch.blockDimZ = 1;
    p->launch.sharedMemBytes = static_cast<unsigned>(p->shape.smem_bytes);
    p->launch_attr[0].id = CU_LAUNCH_ATTRIBUTE_PROGRAMMATIC_STREAM_SERIALIZATION;
    p->launch_attr[0].value.programmaticStreamSerializationAllowed = 1;
    p->launch_attr[1].id = CU_LAUNCH_ATTRIBUTE_CLUSTER_DIMENSION;
    p->launch_attr[1].value.clusterDim.x = static_cast<unsigned>(p->shape.cluster);
    p->launch_attr[1].value.clusterDim.y = 1;
    p->launch_attr[1].value.clusterDim.z = 1;
    p->launch.attrs = p->launch_attr;
    p->launch.numAttrs = (cfg.cta_pair || p->shape.cluster > 1) ? 2 : 1;

    if (dtype == GEMM_I8_I32 && M > 0 && N > 0 && K > 0) {
        st = encode_operand_map(&p->map_a, p->d_a16, M, K,
                                kp.a_half ? gbg::kBM / 2 : gbg::kBM / kp.mcast, a_mn_major(layout),
                                CU_TENSOR_MAP_DATA_TYPE_FLOAT16, cfg.kblocks_per_stage);
        if (st == GEMM_OK)
            st = encode_operand_map(&p->map_b, p->d_b16, N, K,
                                    cfg.cta_pair ? cfg.block_n / 2 : cfg.block_n,
                                    b_mn_major(layout), CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                    cfg.kblocks_per_stage);
        if (st != GEMM_OK) {
            cudaFree(p->dmem);
            delete p;
            return st;
        }
        p->map_a_valid = p->map_b_valid = true;
    }
    *out = p;
    return GEMM_OK;
}

}  // namespace

namespace gbg {

namespace {

const void* variant(int bn, int stages, int out, int pair, int form, size_t* smem,
                    cudaError_t* st) {
    switch (out) {
        case kOutF16:
            return pair ? gemm_variant_pair<kOutF16>(bn, stages, form, smem, st)
                        : gemm_variant_one_sm<kOutF16>(bn, stages, form, smem, st);
        case kOutBF16:
            return pair ? gemm_variant_pair<kOutBF16>(bn, stages, form, smem, st)
                        : gemm_variant_one_sm<kOutBF16>(bn, stages, form, smem, st);
        case kOutI32:
            return pair ? gemm_variant_pair<kOutI32>(bn, stages, form, smem, st)
                        : gemm_variant_one_sm<kOutI32>(bn, stages, form, smem, st);
        default:
            if (smem) *st = cudaErrorInvalidValue;
            return nullptr;
    }
}

}  // namespace

cudaError_t gemm_prepare(int bn, int stages, int out, int pair, int form, size_t* smem_bytes) {
    cudaError_t st = cudaErrorInvalidValue;
    const void* fn = variant(bn, stages, out, pair, form, smem_bytes, &st);
    return fn ? st : cudaErrorInvalidValue;
}

const void* gemm_kernel_ptr(int bn, int stages, int out, int pair, int form) {
    return variant(bn, stages, out, pair, form, nullptr, nullptr);
}

cudaError_t gemm_max_clusters(int bn, int stages, int out, int pair, int form,
                              const LaunchShape& shape, int* n) {
    const void* fn = gemm_kernel_ptr(bn, stages, out, pair, form);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(shape.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(shape.block));
    cfg.dynamicSmemBytes = shape.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(shape.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, fn, &cfg);
}

}  // namespace gbg

extern "C" {

gemm_status_t gemm_plan_create(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                               gemm_layout_t layout, gemm_plan_t* plan) {
    return create_plan(M, N, K, dtype, layout, nullptr, plan);
}

gemm_status_t gemm_plan_create_with_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                           gemm_layout_t layout, const gemm_config_t* config,
                                           gemm_plan_t* plan) {
    if (!config) return GEMM_ERR_INVALID_ARG;
    return create_plan(M, N, K, dtype, layout, config, plan);
}

gemm_status_t gemm_run(gemm_plan_t p, const void* A, const void* B, void* C, void* stream_ptr) {
    return gemm_run_bias_act(p, A, B, C, nullptr, GEMM_ACT_NONE, stream_ptr);
}

gemm_status_t gemm_run_bias_act(gemm_plan_t p, const void* A, const void* B, void* C,
                                const float* bias, gemm_activation_t act, void* stream_ptr) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (act < GEMM_ACT_NONE || act > GEMM_ACT_SILU) return GEMM_ERR_INVALID_ARG;
    if (p->dtype == GEMM_I8_I32 && (bias != nullptr || act != GEMM_ACT_NONE))
        return GEMM_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(bias) & 15u) return GEMM_ERR_ALIGNMENT;
    if (p->M == 0 || p->N == 0) return GEMM_OK;
    if (!C || (p->K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 15u)
        return GEMM_ERR_ALIGNMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (dev != p->device) return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_ptr);
    const int64_t out_bytes = p->M * p->N * (p->dtype == GEMM_I8_I32 ? 4 : 2);

    if (p->K == 0) {
        const cudaError_t e =
            bias ? gbg::launch_fill_bias_act(C, p->M, p->N, bias, static_cast<int>(act),
                                             p->dtype == GEMM_BF16 ? 1 : 0, p->num_sms, stream)
                 : gbg::launch_zero_fill(C, out_bytes, p->num_sms, stream);   // act(0) = 0
        if (e != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        return GEMM_OK;
    }

    if (p->dtype == GEMM_I8_I32) {
        if (gbg::launch_widen_i8(static_cast<const int8_t*>(A), p->M * p->K,
                                 static_cast<const int8_t*>(B), p->N * p->K, p->d_a16, p->d_b16,
                                 p->num_sms, stream) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    } else {
        const CUtensorMapDataType dt = operand_type(p->dtype);
        if (!p->map_a_valid || p->map_a_src != A) {
            p->map_a_valid = false;
            const gemm_status_t st =
                encode_operand_map(&p->map_a, A, p->M, p->K,
                                   p->kp.a_half ? gbg::kBM / 2 : gbg::kBM / p->kp.mcast,
                                   a_mn_major(p->layout), dt, p->cfg.kblocks_per_stage);
            if (st != GEMM_OK) return st;
            p->map_a_src = A;
            p->map_a_valid = true;
        }
        if (!p->map_b_valid || p->map_b_src != B) {
            p->map_b_valid = false;
            // an SM pair loads half of the tile's B rows per CTA
            const int b_rows = p->cfg.cta_pair ? p->cfg.block_n / 2 : p->cfg.block_n;
            const gemm_status_t st =
                encode_operand_map(&p->map_b, B, p->N, p->K, b_rows, b_mn_major(p->layout), dt,
                                   p->cfg.kblocks_per_stage);
            if (st != GEMM_OK) return st;
            p->map_b_src = B;
            p->map_b_valid = true;
        }
    }
    if (!p->map_c_valid || p->map_c_src != C) {
        p->map_c_valid = false;
        const gemm_status_t st = encode_output(&p->map_c, C, p->M, p->N, p->dtype);
        if (st != GEMM_OK) return st;
        p->map_c_src = C;
        p->map_c_valid = true;
    }
    p->kp.C = C;
    p->kp.bias = bias;
    p->kp.act = static_cast<int32_t>(act);
    void* args[4] = {&p->map_a, &p->map_b, &p->map_c, &p->kp};
    p->launch.hStream = reinterpret_cast<CUstream>(stream);
    // (the plain forms compile the fused epilogue out)
    const CUfunction fn = (bias != nullptr || act != GEMM_ACT_NONE) ? p->fn_epilogue : p->fn;
    CUresult r = launch_fn()(&p->launch, fn, args, nullptr);
    if (r == CUDA_ERROR_INVALID_CONTEXT && cudaSetDevice(p->device) == cudaSuccess)
        r = launch_fn()(&p->launch, fn, args, nullptr);   // a thread without a current context
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

gemm_status_t gemm_plan_check(gemm_plan_t p, void* stream_ptr) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_ptr)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    int32_t word = 0;
    if (cudaMemcpy(&word, p->d_error, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (word != 0) {
        const int32_t zero = 0;
        cudaMemcpy(p->d_error, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t p) {
    if (!p) return GEMM_OK;
    gemm_status_t st = GEMM_OK;
    if (p->dmem && cudaFree(p->dmem) != cudaSuccess) {
        cudaGetLastError();
        st = GEMM_ERR_CUDA;
    }
    delete p;
    return st;
}

gemm_status_t gemm_plan_get_config(gemm_plan_t p, gemm_config_t* config) {
    if (!p || !config) return GEMM_ERR_INVALID_ARG;
    *config = p->cfg;
    return GEMM_OK;
}

gemm_status_t gemm_plan_get_launch(gemm_plan_t p, int32_t* grid, int32_t* cluster,
                                   int32_t* max_active_clusters) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    if (grid) *grid = p->shape.grid;
    if (cluster) *cluster = p->shape.cluster;
    if (max_active_clusters) {
        int n = 0;
        int prev = 0;
        cudaGetDevice(&prev);
        if (prev != p->device) cudaSetDevice(p->device);
        if (gbg::gemm_max_clusters(p->cfg.block_n, p->cfg.stages, p->out_kind, p->cfg.cta_pair,
                                   p->form, p->shape, &n) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        if (prev != p->device) cudaSetDevice(prev);
        *max_active_clusters = n;
    }
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_timeout(gemm_plan_t p, uint64_t ns) {
    if (!p) return GEMM_ERR_INVALID_ARG;
    p->kp.timeout_ns = ns ? ns : kDefaultTimeoutNs;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_wait_test(gemm_plan_t p, uint32_t extra_bytes) {
    if (!p || extra_bytes > 4096 || (extra_bytes & 15u)) return GEMM_ERR_INVALID_ARG;
    p->kp.tx_extra = extra_bytes;
    return GEMM_OK;
}

gemm_status_t gemm_select_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 int32_t num_sms, gemm_config_t* config) {
    if (!config || num_sms < 1) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate_shape(M, N, K, dtype, GEMM_LAYOUT_TN);
    if (st != GEMM_OK) return st;
    int32_t per = 0;
    return normalise_config(M, N, K, dtype, gbg::select_config(M, N, K, dtype, num_sms), config, &per);
}

gemm_status_t gemm_tile_coords(int64_t m_blocks, int64_t n_blocks, int32_t raster_group,
                               int64_t tile, int64_t* m_blk, int64_t* n_blk) {
    if (!m_blk || !n_blk || m_blocks < 1 || n_blocks < 1 || raster_group < 1 || tile < 0 ||
        m_blocks * n_blocks > INT32_MAX || tile >= m_blocks * n_blocks)
        return GEMM_ERR_INVALID_ARG;
    // the kernels' multiply-shift evaluation of the raster (a band taller than
    // the grid is the whole grid)
    const int32_t g = raster_group < m_blocks ? raster_group : static_cast<int32_t>(m_blocks);
    const gbg::RasterDiv rd = gbg::make_raster_div(static_cast<int32_t>(m_blocks),
                                                   static_cast<int32_t>(n_blocks), g);
    int32_t m = 0, n = 0;
    gbg::raster_tile_fast(static_cast<int32_t>(m_blocks), rd, static_cast<int32_t>(tile), &m, &n);
    *m_blk = m;
    *n_blk = n;
    return GEMM_OK;
}

gemm_status_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                   const gemm_config_t* config, size_t* bytes) {
    if (!config || !bytes) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate_shape(M, N, K, dtype, GEMM_LAYOUT_TN);
    if (st != GEMM_OK) return st;
    gemm_config_t c;
    int32_t per = 0;
    st = normalise_config(M, N, K, dtype, *config, &c, &per);
    if (st != GEMM_OK) return st;
    *bytes = plan_memory(M, N, K, dtype, c).total;
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: unsupported dtype or layout";
        case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT: pointer or row stride not 16-byte aligned";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no CUDA device";
        case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: device is not sm_103";
        case GEMM_ERR_OOM: return "GEMM_ERR_OOM: device allocation failed";
        case GEMM_ERR_TENSORMAP: return "GEMM_ERR_TENSORMAP: tensor map encoding failed";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch failed";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a kernel wait ran out";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA runtime error";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: split-K partials exceed the fixed 16 MiB scratch of "
                   "gemm_run_splitk_noalloc";
        default: return "unknown gemm_status_t";
    }
}

int32_t gemm_abi_version(void) { return GEMM_ABI_VERSION; }

gemm_status_t gemm_launch_empty(int32_t grid, void* stream) {
    if (grid < 1) return GEMM_ERR_INVALID_ARG;
    if (gbg::launch_empty(grid, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // extern "C"
