// gemm_kernel.cuh -- persistent, warp-specialised TN GEMM for sm_103a (GB300).
//
//   C[M,N] = A[M,K] * B[N,K]^T        A, B K-contiguous; C N-contiguous.
//
// One CTA per SM, 192 threads in three roles:
//   warp 0      TMA producer: one elected thread streams 128 x 64 A tiles and
//               BN x 64 B tiles into a STAGES-deep shared-memory ring with
//               cp.async.bulk.tensor (128-byte swizzle); each slot's mbarrier
//               counts the landed bytes (expect_tx / complete_tx).
//   warp 1      TMEM owner + MMA issuer: one elected thread issues
//               tcgen05.mma (kind::f16, M=128, N=BN, K=16) into a TMEM fp32
//               accumulator and returns each ring slot with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4) ..), convert, store.  The accumulator is double
//               buffered in TMEM so the epilogue of one tile runs under the
//               main loop of the next.
//
// This is the GB300 counterpart of the warp-specialised producer/consumer
// design in "H100 GEMM L2驻留优化：warp-specialized TMA异步拷贝与RL调优策略"
// (paragraph on warp specialisation and the three-way overlap; lists "TMA
// Descriptor", "Async Pipeline"), with WGMMA replaced by a single-thread
// tcgen05.mma issuer and register accumulators replaced by TMEM.  The TMA
// protocol (elected issuing thread, __grid_constant__ tensor maps, mbarrier
// byte accounting for loads, zero fill outside the tensor) follows "B-08.
// Hopper TMA：从单线程 Bulk Copy 到吞吐墙", sections 3.1 and 3.2.
//
// Integer mode (OUT == kOutI32): operands are int8 values already widened to
// fp16 (exact); the MMA accumulates fp32 over chunks of at most `chunk_kb`
// k-blocks, short enough that every partial sum is an integer below 2^24 in
// magnitude and therefore exact in fp32; the epilogue rounds each chunk to
// int32 and sums the chunks in integer registers.
//
// Every wait is bounded (globaltimer); on expiry the thread records a site code
// in the error word, raises a CTA-wide abort flag, and all roles unwind to the
// common exit, which waits for in-flight copies and MMAs and frees TMEM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gemm_kernel_params.h"
#include "gemm_sched.h"

namespace gbg {

// KS = 64-wide k-blocks per ring slot.  A slot's copies complete on one barrier
// phase, and the copy engine turns a phase of one A and one B box around in
// ~0.24 us per SM for boxes up to 32 KiB (measured on GB300), so with KS = 2 or
// 4 the narrow tiles load each operand's KS k-blocks as one 3-D box (operand
// maps viewed as 64 elements x rows x k-blocks) and stream faster.
template <int BN, int STAGES, int KS = 1>
struct SmemLayout {
    static constexpr int kBSubBytes = BN * kBK * 2;              // one k-block of B
    static constexpr int kASlotBytes = KS * kATileBytes;         // A part of a slot
    static constexpr int kBTileBytes = KS * kBSubBytes;          // B part of a slot
    static constexpr int kStageBytes = kASlotBytes + kBTileBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    // Epilogue staging for TMA stores: per epilogue warp two 32-row x 128-byte
    // buffers (128-byte swizzle, 1024-byte aligned).
    static constexpr int kStoreBufBytes = 32 * 128;
    static constexpr int kStagingBytes = kEpiWarps * 2 * kStoreBufBytes;
    static constexpr int kCtlBytes = 256;
    static constexpr int kBiasBytes = kEpiWarps * kBiasSlotBytes;   // after the control block
    static constexpr int kTotal =
        1024 /* alignment slack */ + kRingBytes + kStagingBytes + kCtlBytes + kBiasBytes;
    static_assert(kTotal <= 232448, "exceeds the 227 KiB a CTA may use");
    static_assert(kBTileBytes % 1024 == 0, "128B-swizzle tiles must stay 1024-byte aligned");
    static_assert(STAGES * 16 + 5 * 8 + 16 <= kCtlBytes, "control block overflow");
};

// Control block after the ring.
template <int STAGES>
struct alignas(8) SharedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
    int32_t splitk_last;
};

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool elect_one_sync() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t"
        ".reg .b32 rx;\n\t"
        ".reg .pred px;\n\t"
        "elect.sync rx|px, %1;\n\t"
        "@px mov.s32 %0, 1;\n\t"
        "}"
        : "+r"(pred)
        : "r"(0xffffffffu));
    return pred != 0;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Suspend-time hint of the barrier polls, in ns: measured 10-15% faster
// k-block turnaround on mid-size shapes than the default time limit (the
// hint bounds how long a polling thread may sleep before it looks again).
constexpr uint32_t kWaitHintNs = 32;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "n"(kWaitHintNs)
        : "memory");
    return done != 0;
}

struct Watch {
    volatile int32_t* abort;   // CTA-wide abort flag (shared memory)
    int32_t* error_word;       // plan error word (global memory)
    uint64_t timeout_ns;
};

// Wait until the barrier phase with `parity` has completed.  Returns false if
// the CTA is aborting or the wait ran out (then it records `site`).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Watch& w,
                                           int32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 31u) == 0) {
            if (*w.abort) return false;
            if (global_timer_ns() - t0 > w.timeout_ns) {
                *w.abort = 1;
                atomicCAS(w.error_word, 0, site);
                return false;
            }
        }
    }
}

// Bounded wait used only while unwinding (ignores the abort flag).
__device__ __forceinline__ bool wait_phase_unwind(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Warm L2 with a tile a later tma_load_2d will read (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// 3-D forms for an operand map viewed as (64 elements, rows, k-blocks): one copy
// brings several consecutive 64-wide k-blocks of a tile, stacked k-block-major
// in shared memory (the same image as one 2-D copy per k-block).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t x, int32_t y,
                                                   int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Shared -> global tiled store, tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all committed groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, M=128, N=BN, K=16, fp32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// TMA load delivered to the same shared-memory offset (and barrier offset) in
// every CTA of `cta_mask` within the cluster.
__device__ __forceinline__ void tma_load_2d_mcast(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                  int32_t x, int32_t y, uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(cta_mask)
        : "memory");
}

// As umma_commit, arriving on the barrier at this offset in every CTA of `cta_mask`.
__device__ __forceinline__ void umma_commit_mcast(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms
// stacked at a 1024-byte stride.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)   // start address / 16
           | (static_cast<uint64_t>(1) << 16)                // leading byte offset (unused here)
           | (static_cast<uint64_t>(1024 >> 4) << 32)        // stride byte offset: 8 rows * 128 B
           | (static_cast<uint64_t>(1) << 46)                // descriptor version (tcgen05)
           | (static_cast<uint64_t>(2) << 61);               // swizzle mode: 128 B
}

// Shared-memory descriptor for an MN-major operand tile written by TMA as
// 64-element (128-byte) wide blocks of KS*64 K-rows (KS*8 KiB each, 128-byte
// swizzle): 8-row K groups 1024 bytes apart (stride byte offset), 64-element MN
// blocks KS*8 KiB apart (leading byte offset).
template <int KS = 1>
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)
           | (static_cast<uint64_t>((KS * 8192) >> 4) << 16)  // leading byte offset: next 64 MN
           | (static_cast<uint64_t>(1024 >> 4) << 32)         // stride byte offset: next 8 K rows
           | (static_cast<uint64_t>(1) << 46)
           | (static_cast<uint64_t>(2) << 61);
}
template <int KS = 1>
__device__ __forceinline__ uint64_t operand_desc(uint32_t saddr, int32_t mn_major) {
    return mn_major ? sw128_mnmajor_desc<KS>(saddr) : sw128_kmajor_desc(saddr);
}
// Offset of k-block j of a slot within an operand's part of the slot: K-major
// parts hold KS whole rows x 64 tiles (tile_bytes each); MN-major parts hold
// 64-element blocks of KS*64 K-rows, where k-block j starts 64 K-rows (8 KiB) in.
__device__ __forceinline__ uint32_t kblock_offset(int32_t mn_major, uint32_t tile_bytes, int j) {
    return static_cast<uint32_t>(j) * (mn_major ? 8192u : tile_bytes);
}
// Descriptor advance per K=16 MMA: 32 bytes along a K-major row, or 16 rows of
// 128 bytes of an MN-major tile (start address is encoded >> 4).
__device__ __forceinline__ uint32_t desc_k_step(int32_t mn_major) { return mn_major ? 128u : 2u; }

// One operand tile (`rows` rows of M or N by 64 K) of k-block kb into `dst`:
// K-major = one box {64 K, rows}; MN-major = rows/64 boxes {64 MN, 64 K}, 8 KiB apart.
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int32_t kb, int32_t row0, int32_t rows,
                                             int32_t mn_major) {
    if (!mn_major) {
        tma_load_2d(dst, map, bar, kb * kBK, row0);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i)
        tma_load_2d(dst + static_cast<uint32_t>(i) * 8192u, map, bar, row0 + i * 64, kb * kBK);
}
__device__ __forceinline__ void prefetch_operand(const CUtensorMap* map, int32_t kb, int32_t row0,
                                                 int32_t rows, int32_t mn_major) {
    if (!mn_major) {
        tma_prefetch_l2_2d(map, kb * kBK, row0);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i) tma_prefetch_l2_2d(map, row0 + i * 64, kb * kBK);
}

// KS consecutive k-blocks kb .. kb+KS-1 of an operand tile for a multi-k-block
// slot: K-major = one 3-D box {64, rows, KS} of the (64, rows, K/64) view;
// MN-major = rows/64 boxes {64 MN, KS*64 K} (the map's box is KS*64 K-rows
// high), KS*8 KiB apart.
template <int KS>
__device__ __forceinline__ void load_operand_kb(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                int32_t kb, int32_t row0, int32_t rows,
                                                int32_t mn_major) {
    if (!mn_major) {
        tma_load_3d(dst, map, bar, 0, row0, kb);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i)
        tma_load_2d(dst + static_cast<uint32_t>(i * KS) * 8192u, map, bar, row0 + i * 64, kb * kBK);
}
__device__ __forceinline__ void prefetch_operand_kb(const CUtensorMap* map, int32_t kb, int32_t row0,
                                                    int32_t rows, int32_t mn_major) {
    if (!mn_major) {
        tma_prefetch_l2_3d(map, 0, row0, kb);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i) tma_prefetch_l2_2d(map, row0 + i * 64, kb * kBK);
}

// 32 lanes x 32 consecutive 32-bit TMEM columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint4 ld_cg_u4(const void* p) {
    return __ldcg(reinterpret_cast<const uint4*>(p));
}

// ----------------------------------------------------------------------------
// epilogue helpers: one thread owns one output row and 32 consecutive columns
// ----------------------------------------------------------------------------
template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (OUT == kOutF16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// Fused epilogue of a linear layer, in fp32 before the output conversion:
// x = act(x + bias[col]).
// The epilogue's activation, chosen at compile time: the kernel dispatches on
// the plan's activation once per group of columns, not per element.
template <int ACT>
__device__ __forceinline__ float act_fn(float x) {
    if constexpr (ACT == 1) {
        return fmaxf(x, 0.0f);
    } else if constexpr (ACT == 2) {
        return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));   // x * Phi(x)
    } else if constexpr (ACT == 3) {
        // x * sigmoid(x); the fast exponential and divide are far inside the
        // epilogue tolerance and keep the four epilogue warps ahead of the MMA
        return __fdividef(x, 1.0f + __expf(-x));
    } else {
        return x;
    }
}

// v holds fp32 bits for columns [col, col + 4*G); N % 8 == 0, so a group of 4
// columns is entirely inside or outside C.  The bias loads are issued together
// before any use.
template <int ACT, int G>
__device__ __forceinline__ void bias_act(uint32_t* v, const float* bias, int32_t N, int32_t col) {
    float4 b[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        b[g] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias != nullptr && col + g * 4 < N)
            b[g] = __ldg(reinterpret_cast<const float4*>(bias + col + g * 4));
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        v[g * 4 + 0] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 0]) + b[g].x));
        v[g * 4 + 1] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 1]) + b[g].y));
        v[g * 4 + 2] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 2]) + b[g].z));
        v[g * 4 + 3] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 3]) + b[g].w));
    }
}

template <int G>
__device__ __forceinline__ void apply_bias_act(uint32_t* v, const KParams& p, int32_t col) {
    if (p.bias == nullptr && p.act == 0) return;
    switch (p.act) {
        case 1: bias_act<1, G>(v, p.bias, p.N, col); break;
        case 2: bias_act<2, G>(v, p.bias, p.N, col); break;
        case 3: bias_act<3, G>(v, p.bias, p.N, col); break;
        default: bias_act<0, G>(v, p.bias, p.N, col); break;
    }
}

// The fused bias of a 64-column chunk, staged in the epilogue warp's shared
// memory slot: each lane fetches two columns one chunk ahead (global latency off
// the chunk's path), the warp writes them to its slot, and the 32-column halves
// read them back four columns per broadcast load.  N % 8 == 0 and col is even:
// both columns are inside or outside C.
__device__ __forceinline__ float2 bias_fetch2(const float* bias, int32_t N, int32_t col) {
    if (bias == nullptr || col >= N) return make_float2(0.f, 0.f);
    return __ldg(reinterpret_cast<const float2*>(bias + col));
}
__device__ __forceinline__ void st_shared_f2(uint32_t saddr, float2 v) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(saddr), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}
template <int ACT, int G>
__device__ __forceinline__ void bias_act_staged(uint32_t* v, uint32_t b_addr) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float4 b = ld_shared_f4(b_addr + static_cast<uint32_t>(g * 16));
        v[g * 4 + 0] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 0]) + b.x));
        v[g * 4 + 1] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 1]) + b.y));
        v[g * 4 + 2] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 2]) + b.z));
        v[g * 4 + 3] = __float_as_uint(act_fn<ACT>(__uint_as_float(v[g * 4 + 3]) + b.w));
    }
}
// v: 4*G columns whose bias values start at shared address b_addr.
template <int G>
__device__ __forceinline__ void apply_bias_act_staged(uint32_t* v, const KParams& p, uint32_t b_addr) {
    switch (p.act) {
        case 1: bias_act_staged<1, G>(v, b_addr); break;
        case 2: bias_act_staged<2, G>(v, b_addr); break;
        case 3: bias_act_staged<3, G>(v, b_addr); break;
        default: bias_act_staged<0, G>(v, b_addr); break;
    }
}

// Store 32 fp32 values (as bits) of row `row`, columns [col, col+32) as fp16/bf16.
template <int OUT>
__device__ __forceinline__ void store_half_row32(void* C, int32_t N, int32_t row, int32_t col,
                                                 const uint32_t (&v)[32]) {
    uint16_t* base = reinterpret_cast<uint16_t*>(C) + static_cast<int64_t>(row) * N;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int32_t c = col + g * 8;
        if (c < N) {   // N % 8 == 0: an 8-column group is entirely in or out
            uint4 q;
            q.x = pack2<OUT>(__uint_as_float(v[g * 8 + 0]), __uint_as_float(v[g * 8 + 1]));
            q.y = pack2<OUT>(__uint_as_float(v[g * 8 + 2]), __uint_as_float(v[g * 8 + 3]));
            q.z = pack2<OUT>(__uint_as_float(v[g * 8 + 4]), __uint_as_float(v[g * 8 + 5]));
            q.w = pack2<OUT>(__uint_as_float(v[g * 8 + 6]), __uint_as_float(v[g * 8 + 7]));
            *reinterpret_cast<uint4*>(base + c) = q;
        }
    }
}

// Store 32 int32 values of row `row`, columns [col, col+32).
__device__ __forceinline__ void store_i32_row32(void* C, int32_t N, int32_t row, int32_t col,
                                                const uint32_t* v) {
    uint32_t* base = reinterpret_cast<uint32_t*>(C) + static_cast<int64_t>(row) * N;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int32_t c = col + g * 4;
        if (c < N) {   // N % 4 == 0
            *reinterpret_cast<uint4*>(base + c) =
                make_uint4(v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]);
        }
    }
}

__device__ __forceinline__ void store_ws32(uint32_t* dst, const uint32_t* v) {
#pragma unroll
    for (int g = 0; g < 8; ++g)
        __stcg(reinterpret_cast<uint4*>(dst) + g,
               make_uint4(v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]));
}

template <int OUT>
__device__ __forceinline__ void add_u4(uint32_t* v, const uint4& q) {
    if constexpr (OUT == kOutI32) {   // integer partials: wrap-around sums (mod 2^32)
        v[0] += q.x;
        v[1] += q.y;
        v[2] += q.z;
        v[3] += q.w;
    } else {
        v[0] = __float_as_uint(__uint_as_float(v[0]) + __uint_as_float(q.x));
        v[1] = __float_as_uint(__uint_as_float(v[1]) + __uint_as_float(q.y));
        v[2] = __float_as_uint(__uint_as_float(v[2]) + __uint_as_float(q.z));
        v[3] = __float_as_uint(__uint_as_float(v[3]) + __uint_as_float(q.w));
    }
}

// v = sum over K slices s = 0..S-1 (in that order) of 32 partial values at
// src + s*slice_stride.  G slices' loads are issued before any is added, so
// G x 128 bytes per thread are in flight.
template <int OUT, int G>
__device__ __forceinline__ void reduce_slices32(const uint32_t* src, int64_t slice_stride,
                                                int32_t S, uint32_t (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0u;   // +0.0f and integer 0 share the bit pattern
    for (int32_t s0 = 0; s0 < S; s0 += G) {
        uint4 q[G][8];
#pragma unroll
        for (int t = 0; t < G; ++t) {
            if (s0 + t < S) {
                const uint32_t* slice = src + (s0 + t) * slice_stride;
#pragma unroll
                for (int g = 0; g < 8; ++g) q[t][g] = ld_cg_u4(slice + g * 4);
            }
        }
#pragma unroll
        for (int t = 0; t < G; ++t) {
            if (s0 + t < S) {
#pragma unroll
                for (int g = 0; g < 8; ++g) add_u4<OUT>(&v[g * 4], q[t][g]);
            }
        }
    }
}

// ---- thread-block cluster / distributed shared memory
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared::cluster address of the same offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint4 ld_dsmem_u4(uint32_t cluster_addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_u4(uint32_t saddr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
// All threads of all CTAs of the cluster; release/acquire orders shared memory.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Partial tile staged in shared memory for the cluster reduction: 128 rows of
// BN 32-bit values, row stride BN+4 words (keeps the row-per-thread writes of a
// warp on distinct banks).
template <int BN>
__device__ __forceinline__ void stage_row32(uint32_t staging, int row, int col, const uint32_t* v) {
    const uint32_t base = staging + static_cast<uint32_t>((row * (BN + 4) + col) * 4);
#pragma unroll
    for (int g = 0; g < 8; ++g)
        st_shared_u4(base + g * 16, make_uint4(v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]));
}

// In-cluster split-K reduction (push, then local sums).  The S K-slices of a
// 128-row block of C sit in S cluster CTAs; CTA "part" o (rank o * rank_stride +
// rank_offset) owns rows [o*128/S, (o+1)*128/S) of the block.  After a cluster
// barrier (every ring idle) each CTA stores each of its fp32 partial rows into
// the owner's receive area, slot = its own slice index; after a second barrier
// every owner sums its S slots in slice order 0..S-1 (fixed order: the same
// result every run) from its own shared memory and writes C.
// Receive area: S slots x 128/S rows x BN words, row stride BN+4 words.
template <int BN>
struct SplitRecv {
    static constexpr int kRowWords = BN + 4;
    static constexpr int kBytes = kBM * kRowWords * 4;
};

__device__ __forceinline__ void st_dsmem_u4(uint32_t cluster_addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr)
                 : "memory");
    return v;
}

// Push phase, S K-slices (S fixed at compile time).  Epilogue warp `quad` sends
// its 32 partial rows [32*quad, 32*quad+32) of K-slice `slice` (from TMEM, or
// for integer outputs from the parked sums at `parked`), 32 columns at a time,
// into the receive areas of the rows' owners.  The values pass through the
// warp's staging buffer (36-word row stride: both passes are free of bank
// conflicts) so that each remote store instruction writes 4 rows x 128
// contiguous bytes instead of 32 scattered 16-byte pieces.  With S known, the
// owner of every group of 4 rows is known too: the warp maps each owner's
// destination once and every later address is that base plus an immediate
// (the loop is issue-bound: one warp per SM sub-partition runs it).
template <int BN, int OUT, int S>
__device__ __forceinline__ void cluster_push(uint32_t recv, uint32_t stg, uint32_t tmem_base,
                                             uint32_t parked, int quad, int lane, int slice,
                                             uint32_t rank_stride, uint32_t rank_offset) {
    constexpr int kRows = kBM / S;                       // rows per owner: 64, 32 or 16
    constexpr int kOwners = kRows >= 32 ? 1 : 32 / kRows;   // owners of one warp's rows
    constexpr int kSpan = 32 / kOwners;                  // warp rows per owner
    constexpr int kRowB = SplitRecv<BN>::kRowWords * 4;
    const int ch = lane & 7;
    const int sub = lane >> 3;
    uint32_t dst[kOwners];
#pragma unroll
    for (int k = 0; k < kOwners; ++k) {
        const int row0 = quad * 32 + k * kSpan;
        const int owner = row0 / kRows;
        const uint32_t local =
            recv + static_cast<uint32_t>((slice * kRows + row0 % kRows + sub) * kRowB + ch * 16);
        dst[k] = map_to_rank(local, static_cast<uint32_t>(owner) * rank_stride + rank_offset);
    }
    const uint32_t stg_w = stg + static_cast<uint32_t>(lane * 36 * 4);
    const uint32_t stg_r = stg + static_cast<uint32_t>((sub * 36 + 4 * ch) * 4);
    const uint32_t src_t = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t src_p = parked + static_cast<uint32_t>((quad * 32 + lane) * (BN + 4) * 4);
    // 32 partial values of this thread's row, columns [32j, 32j+32)
    auto fetch = [&](int j, uint32_t (&v)[32]) {
        if constexpr (OUT == kOutI32) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const uint4 q = ld_shared_u4(src_p + static_cast<uint32_t>(j * 128 + g * 16));
                v[g * 4 + 0] = q.x;
                v[g * 4 + 1] = q.y;
                v[g * 4 + 2] = q.z;
                v[g * 4 + 3] = q.w;
            }
        } else {
            tmem_ld_32x32b_x32(src_t + static_cast<uint32_t>(j * 32), v);
        }
    };
    // (fully unrolled: no loop-carried copy of v can be placed between an
    // asynchronous TMEM read and its wait)
    uint32_t v[32];
    fetch(0, v);
#pragma unroll
    for (int j = 0; j < BN / 32; ++j) {
        if constexpr (OUT != kOutI32) tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 8; ++g)
            st_shared_u4(stg_w + g * 16,
                         make_uint4(v[g * 4 + 0], v[g * 4 + 1], v[g * 4 + 2], v[g * 4 + 3]));
        __syncwarp();
        // the next block's TMEM read overlaps this block's sends
        if (j + 1 < BN / 32) fetch(j + 1, v);
        uint4 q[8];   // rows 4s + sub of the warp: all loads before the first send
#pragma unroll
        for (int s = 0; s < 8; ++s) q[s] = ld_shared_u4(stg_r + static_cast<uint32_t>(s * 4 * 36 * 4));
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int k = (4 * s) / kSpan;
            st_dsmem_u4(dst[k] + static_cast<uint32_t>((4 * s - k * kSpan) * kRowB + j * 128), q[s]);
        }
        __syncwarp();   // the staging buffer is rewritten in the next round
    }
}

template <int BN, int OUT, int kMaxS>
__device__ __forceinline__ void cluster_push_any(int S, uint32_t recv, uint32_t stg,
                                                 uint32_t tmem_base, uint32_t parked, int quad,
                                                 int lane, int slice, uint32_t rank_stride,
                                                 uint32_t rank_offset) {
    if (S == 2)
        cluster_push<BN, OUT, 2>(recv, stg, tmem_base, parked, quad, lane, slice, rank_stride,
                                 rank_offset);
    else if (S == 4)
        cluster_push<BN, OUT, 4>(recv, stg, tmem_base, parked, quad, lane, slice, rank_stride,
                                 rank_offset);
    else if constexpr (kMaxS >= 8)
        cluster_push<BN, OUT, 8>(recv, stg, tmem_base, parked, quad, lane, slice, rank_stride,
                                 rank_offset);
}

// The owner's half, S slices (compile-time): sum its S slots in slice order
// 0..S-1, apply the epilogue, store rows [part*128/S, (part+1)*128/S) of the
// block whose first global row is block_row.  The 128 epilogue threads take
// consecutive 4-column groups (coalesced stores); a thread's groups are
// 128/(BN/4) rows apart, so every shared-memory address is the thread's base
// plus an immediate, and a batch issues up to 16 loads before its first add.
template <int BN, int OUT, int S, bool EPI>
__device__ __forceinline__ void cluster_sum_store_s(const KParams& p, int32_t block_row,
                                                    int32_t col_base, int part, uint32_t recv,
                                                    int tid) {
    constexpr int kRows = kBM / S;
    constexpr int kVec = BN / 4;                      // 4-column groups per row
    constexpr int kRowStep = kEpiWarps * 32 / kVec;   // rows between a thread's groups
    constexpr int kG = kRows / kRowStep;              // groups per thread
    constexpr int kB = (16 / S) < kG ? (16 / S) : kG;  // groups per batch
    constexpr uint32_t kSlot = kRows * SplitRecv<BN>::kRowWords * 4;
    constexpr uint32_t kStepB = kRowStep * SplitRecv<BN>::kRowWords * 4;
    static_assert(kG % kB == 0, "whole batches");
    const int c4 = (tid % kVec) * 4;
    const int lr0 = tid / kVec;
    const int32_t gcol = col_base + c4;
    if (gcol >= p.N) return;
    const int32_t grow0 = block_row + part * kRows + lr0;
    const uint32_t src = recv + static_cast<uint32_t>((lr0 * SplitRecv<BN>::kRowWords + c4) * 4);
    const int64_t step = static_cast<int64_t>(kRowStep) * p.N;
    const int64_t idx0 = static_cast<int64_t>(grow0) * p.N + gcol;
#pragma unroll
    for (int b = 0; b < kG; b += kB) {
        if (grow0 + b * kRowStep >= p.M) break;   // later groups lie further down
        uint4 q[kB][S];
#pragma unroll
        for (int i = 0; i < kB; ++i)
#pragma unroll
            for (int s = 0; s < S; ++s)
                q[i][s] = ld_shared_u4(src + (b + i) * kStepB + s * kSlot);
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            if (grow0 + (b + i) * kRowStep >= p.M) break;
            uint32_t v[4] = {q[i][0].x, q[i][0].y, q[i][0].z, q[i][0].w};
#pragma unroll
            for (int s = 1; s < S; ++s) add_u4<OUT>(v, q[i][s]);
            const int64_t idx = idx0 + (b + i) * step;
            if constexpr (OUT == kOutI32) {
                *reinterpret_cast<uint4*>(reinterpret_cast<uint32_t*>(p.C) + idx) =
                    make_uint4(v[0], v[1], v[2], v[3]);
            } else {
                if constexpr (EPI) apply_bias_act<1>(v, p, gcol);
                uint2 h;
                h.x = pack2<OUT>(__uint_as_float(v[0]), __uint_as_float(v[1]));
                h.y = pack2<OUT>(__uint_as_float(v[2]), __uint_as_float(v[3]));
                *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.C) + idx) = h;
            }
        }
    }
}

template <int BN, int OUT, int S>
__device__ __forceinline__ void cluster_sum_store_e(const KParams& p, int32_t block_row,
                                                    int32_t col_base, int part, uint32_t recv,
                                                    int tid) {
    // (the loop without the bias/activation code when the plan has none)
    if (OUT == kOutI32 || (p.bias == nullptr && p.act == 0))
        cluster_sum_store_s<BN, OUT, S, false>(p, block_row, col_base, part, recv, tid);
    else
        cluster_sum_store_s<BN, OUT, S, OUT != kOutI32>(p, block_row, col_base, part, recv, tid);
}

template <int BN, int OUT, int kMaxS>
__device__ __forceinline__ void cluster_sum_store(const KParams& p, int32_t block_row,
                                                  int32_t col_base, int part, uint32_t recv,
                                                  int tid) {
    if (p.split_k == 2)
        cluster_sum_store_e<BN, OUT, 2>(p, block_row, col_base, part, recv, tid);
    else if (p.split_k == 4)
        cluster_sum_store_e<BN, OUT, 4>(p, block_row, col_base, part, recv, tid);
    else if constexpr (kMaxS >= 8)
        cluster_sum_store_e<BN, OUT, 8>(p, block_row, col_base, part, recv, tid);
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Write `nchunks` 16-byte chunks (4 words each) of row `row` of a 32-row x
// 128-byte store buffer, starting at logical chunk c0, in the 128-byte swizzle
// the C tensor map uses (chunk c of row r sits at chunk c ^ (r & 7)): the 8
// rows of a quarter-warp hit 8 distinct bank groups.
__device__ __forceinline__ void stage_store_row(uint32_t buf, int row, int c0, const uint32_t* w,
                                                int nchunks) {
    const uint32_t row_base = buf + static_cast<uint32_t>(row) * 128u;
#pragma unroll
    for (int i = 0; i < nchunks; ++i) {
        const uint32_t chunk = static_cast<uint32_t>((c0 + i) ^ (row & 7));
        st_shared_u4(row_base + chunk * 16u,
                     make_uint4(w[i * 4 + 0], w[i * 4 + 1], w[i * 4 + 2], w[i * 4 + 3]));
    }
}

// Persistent iteration space of this CTA: units blockIdx.x, +gridDim.x, ... or,
// with A multicast, tile groups cluster_id, +num_clusters, ... shared by the
// CTAs of a cluster.
struct UnitIter {
    int32_t first, stride;
};
__device__ __forceinline__ UnitIter unit_iter(const KParams& p) {
    return UnitIter{static_cast<int32_t>(blockIdx.x >> p.mcast_shift),
                    static_cast<int32_t>(gridDim.x >> p.mcast_shift)};
}
// Coordinates of unit u for this CTA.  With multicast, unit u is a group of
// mcast adjacent n-blocks of one m-block, this CTA taking the one of its
// cluster rank; a tile past N loads zeros and stores nothing.
__device__ __forceinline__ UnitCoord unit_at(const KParams& p, int32_t u) {
    UnitCoord c = unit_coord_fast(u, p);   // with multicast: tile group u (split_k is 1)
    if (p.mcast > 1)
        c.n_blk = c.n_blk * p.mcast + static_cast<int32_t>(blockIdx.x & (p.mcast - 1));
    return c;
}

// The kernel's parameters in compiled form FORM (see KernelForm): the fields the
// form fixes are constants, so the paths of the other modes compile away.  A
// launch's chain from the dependency release to its last exit is ~0.75 us
// shorter in the plain form for a one-tile GEMM (2.33 -> 1.58 us, 64x64x64 on
// GB300: the code each role runs first after the wait is smaller and has no
// mode branches).
template <int FORM>
__device__ __forceinline__ KParams form_params(const KParams& in) {
    if constexpr (FORM == kFormGeneral) {
        return in;
    } else {
        KParams p = in;
        p.mcast = 1;
        p.mcast_shift = 0;
        p.direct_store = 0;
        p.l2_prefetch = 0;
        p.a_mn_major = 0;
        p.b_mn_major = 0;
        if constexpr (FORM != kFormEpilogue) {
            // a call with a fused bias or activation launches the epilogue or the
            // general form
            p.bias = nullptr;
            p.act = 0;
        }
        if constexpr (FORM == kFormPlain || FORM == kFormEpilogue) {
            p.split_k = 1;
            p.cluster_split = 0;
        } else {
            p.cluster_split = 1;   // split_k (2, 4 or 8) stays a run-time value
        }
        return p;
    }
}

// ----------------------------------------------------------------------------
// the kernel
// ----------------------------------------------------------------------------
// KS > 1: each K-major operand's map is the 3-D view (the host guarantees it
// and K % 64 == 0; multicast is not combined with it).  FORM: a KernelForm whose
// fixed fields match the plan's (the host picks the form).
template <int BN, int STAGES, int OUT, int KS = 1, int FORM = kFormGeneral>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tn_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, const KParams p_in) {
    const KParams p = form_params<FORM>(p_in);
    using L = SmemLayout<BN, STAGES, KS>;
    static_assert(KS == 1 || KS == 2 || KS == 4, "k-blocks per ring slot");
    static_assert((OUT == kOutI32 ? 2 : 1) * SplitRecv<BN>::kBytes <= L::kRingBytes,
                  "split-K receive area (and parked integer sums) must fit in the ring");
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static_assert(OUT != kOutI32 || BN <= 128, "integer mode keeps BN int32 sums in registers");
    constexpr uint32_t kTmemCols = 2 * BN;   // two accumulator buffers; 128/256/512 columns
    constexpr uint32_t kStageTx = L::kStageBytes;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t ring = smem_addr(smem);                       // A slots, then B slots
    const uint32_t ring_b = ring + STAGES * L::kASlotBytes;
    const uint32_t staging = ring + L::kRingBytes;              // epilogue store buffers
    SharedCtl<STAGES>* ctl =
        reinterpret_cast<SharedCtl<STAGES>*>(smem + L::kRingBytes + L::kStagingBytes);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        prefetch_tmap(&tmap_c);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            // with A multicast a slot is free only once every CTA of the cluster
            // has consumed it (each one's MMA commit arrives here)
            mbar_init(smem_addr(&ctl->empty[s]), p.mcast > 1 ? p.mcast : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl->tmem_full[b]), 1);
            mbar_init(smem_addr(&ctl->tmem_empty[b]), kEpiWarps);
        }
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort = 0;
        ctl->splitk_last = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    if (p.mcast > 1)
        cluster_sync_all();   // peers' copies and commits target this CTA's barriers
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    // Programmatic dependent launch: the set-up above may overlap the previous
    // kernel of the stream; no global memory is touched before that kernel has
    // completed and its writes are visible.  The next kernel may be scheduled
    // from here on (it waits the same way before reading anything we write).
    const UnitIter it = unit_iter(p);
    // This CTA's first unit, worked out while the previous kernel may still run.
    const UnitCoord c_first = unit_at(p, it.first);
    // Plain and cluster split forms: ring slots of the first unit that the copy
    // thread arms before the wait (shared memory only), so that right after it
    // only their copies are issued (kArmedCopy).
    int32_t n_armed = 0;
    if constexpr (kArmedCopy<FORM>) {
        if (warp == 0 && lane == 0 && it.first < p.num_units) {
            const int32_t nslots = (c_first.kb_end - c_first.kb_begin + KS - 1) / KS;
            n_armed = nslots < STAGES ? nslots : STAGES;
            const uint32_t tx = kStageTx - (p.a_half ? KS * 8192u : 0u) + p.tx_extra;
            for (int32_t s = 0; s < n_armed; ++s) mbar_arrive_expect_tx(smem_addr(&ctl->full[s]), tx);
        }
    }
    if (warp == 0 && lane == 0 && it.first < p.num_units) {
        // Warm L2 with this CTA's first k-blocks while the previous kernel drains.
        // Only L2 is touched (the coherence point); the data is read after the
        // wait below, so this cannot observe stale values.
        const UnitCoord c = c_first;
        const int32_t ahead = STAGES * KS > p.l2_prefetch ? STAGES * KS : p.l2_prefetch;
        const int32_t kb_end = c.kb_begin + ahead < c.kb_end ? c.kb_begin + ahead : c.kb_end;
        // with multicast, this CTA's slice of the A tile (its A box is that slice)
        const int32_t a_rows = p.a_half ? kBM / 2 : (kBM >> p.mcast_shift);
        const int32_t a_row0 =
            c.m_blk * kBM + static_cast<int32_t>(blockIdx.x & ((1u << p.mcast_shift) - 1u)) * a_rows;
        for (int32_t kb = c.kb_begin; kb < kb_end; kb += KS) {
            if constexpr (KS > 1) {
                prefetch_operand_kb(&tmap_a, kb, a_row0, a_rows, p.a_mn_major);
                prefetch_operand_kb(&tmap_b, kb, c.n_blk * BN, BN, p.b_mn_major);
            } else {
                prefetch_operand(&tmap_a, kb, a_row0, a_rows, p.a_mn_major);
                prefetch_operand(&tmap_b, kb, c.n_blk * BN, BN, p.b_mn_major);
            }
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();
    const Watch watch{&ctl->abort, p.error_word, p.timeout_ns};
    bool epi_ok = false;   // epilogue: this CTA's accumulator is complete (split-K in the cluster)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if constexpr (kArmedCopy<FORM>) {
            // (no multicast, no L2 prefetch distance, K-contiguous operands)
            if (lane == 0) {   // the thread that armed the first slots
                const uint32_t slot_tx = kStageTx - (p.a_half ? KS * 8192u : 0u) + p.tx_extra;
                auto issue = [&](int stage, int32_t kb, const UnitCoord& c) {
                    const uint32_t full = smem_addr(&ctl->full[stage]);
                    if constexpr (KS > 1) {
                        load_operand_kb<KS>(ring + stage * L::kASlotBytes, &tmap_a, full, kb,
                                            c.m_blk * kBM, p.a_half ? kBM / 2 : kBM, 0);
                        load_operand_kb<KS>(ring_b + stage * L::kBTileBytes, &tmap_b, full, kb,
                                            c.n_blk * BN, BN, 0);
                    } else {
                        load_operand(ring + stage * kATileBytes, &tmap_a, full, kb, c.m_blk * kBM,
                                     p.a_half ? kBM / 2 : kBM, 0);
                        load_operand(ring_b + stage * L::kBTileBytes, &tmap_b, full, kb,
                                     c.n_blk * BN, BN, 0);
                    }
                };
                for (int32_t s = 0; s < n_armed; ++s) issue(s, c_first.kb_begin + s * KS, c_first);
                int stage = n_armed == STAGES ? 0 : n_armed;
                uint32_t phase = n_armed == STAGES ? 1u : 0u;
                int issued = n_armed;
                bool ok = true;
                for (int32_t u = it.first; ok && u < p.num_units; u += it.stride) {
                    const UnitCoord c = u == it.first ? c_first : unit_at(p, u);
                    for (int32_t kb = u == it.first ? c.kb_begin + n_armed * KS : c.kb_begin;
                         kb < c.kb_end; kb += KS) {
                        if (issued >= STAGES &&
                            !wait_phase(smem_addr(&ctl->empty[stage]), phase ^ 1u, watch,
                                        kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(smem_addr(&ctl->full[stage]), slot_tx);
                        issue(stage, kb, c);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                // every copy issued lands before the CTA can exit (see below)
                const int pending = issued < STAGES ? issued : STAGES;
                for (int i = 0; i < pending; ++i) {
                    if (--stage < 0) {
                        stage = STAGES - 1;
                        phase ^= 1u;
                    }
                    wait_phase_unwind(smem_addr(&ctl->full[stage]), phase, 100000000ull);
                }
            }
        } else if (elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int32_t u = it.first; ok && u < p.num_units; u += it.stride) {
                const UnitCoord c = u == it.first ? c_first : unit_at(p, u);
                for (int32_t kb = c.kb_begin; kb < c.kb_end; kb += KS) {
                    const uint32_t full = smem_addr(&ctl->full[stage]);
                    // (the first pass over the ring finds every slot free)
                    if (issued >= STAGES &&
                        !wait_phase(smem_addr(&ctl->empty[stage]), phase ^ 1u, watch,
                                    kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    // (a half-height A tile delivers 8 KiB less per k-block)
                    mbar_arrive_expect_tx(full, kStageTx - (p.a_half ? KS * 8192u : 0u) + p.tx_extra);
                    if constexpr (KS > 1) {
                        // the slot's KS k-blocks of each operand in one copy; a copy
                        // past the end of K is zero-filled and past the slice end is
                        // unused, but always delivers the full box
                        load_operand_kb<KS>(ring + stage * L::kASlotBytes, &tmap_a, full, kb,
                                            c.m_blk * kBM, p.a_half ? kBM / 2 : kBM, p.a_mn_major);
                        load_operand_kb<KS>(ring_b + stage * L::kBTileBytes, &tmap_b, full, kb,
                                            c.n_blk * BN, BN, p.b_mn_major);
                        if (p.l2_prefetch > 0 && kb + p.l2_prefetch < c.kb_end) {
                            prefetch_operand_kb(&tmap_a, kb + p.l2_prefetch, c.m_blk * kBM,
                                                p.a_half ? kBM / 2 : kBM, p.a_mn_major);
                            prefetch_operand_kb(&tmap_b, kb + p.l2_prefetch, c.n_blk * BN, BN,
                                                p.b_mn_major);
                        }
                    } else {
                        if (p.mcast > 1) {
                            // this CTA's 1/mcast of the A tile, delivered to every CTA of
                            // the cluster (the slot's bytes arrive from all of them)
                            const int32_t rank = static_cast<int32_t>(blockIdx.x & (p.mcast - 1));
                            const uint16_t all = static_cast<uint16_t>((1u << p.mcast) - 1u);
                            const uint32_t a_slot = ring + stage * kATileBytes;
                            if (p.a_mn_major) {   // mcast == 2: one 64-row M block each
                                tma_load_2d_mcast(a_slot + static_cast<uint32_t>(rank) * 8192u,
                                                  &tmap_a, full, c.m_blk * kBM + rank * 64, kb * kBK,
                                                  all);
                            } else {
                                const int32_t rows = kBM >> p.mcast_shift;
                                tma_load_2d_mcast(a_slot + static_cast<uint32_t>(rank * rows * 128),
                                                  &tmap_a, full, kb * kBK, c.m_blk * kBM + rank * rows,
                                                  all);
                            }
                        } else {
                            load_operand(ring + stage * kATileBytes, &tmap_a, full, kb, c.m_blk * kBM,
                                         p.a_half ? kBM / 2 : kBM, p.a_mn_major);
                        }
                        load_operand(ring_b + stage * L::kBTileBytes, &tmap_b, full, kb, c.n_blk * BN,
                                     BN, p.b_mn_major);
                        if (p.l2_prefetch > 0 && kb + p.l2_prefetch < c.kb_end) {
                            // warm L2 with a later k-block of this tile (this CTA's A share)
                            const int32_t a_rows = p.a_half ? kBM / 2 : (kBM >> p.mcast_shift);
                            const int32_t a_rank =
                                static_cast<int32_t>(blockIdx.x & ((1u << p.mcast_shift) - 1u));
                            prefetch_operand(&tmap_a, kb + p.l2_prefetch,
                                             c.m_blk * kBM + a_rank * a_rows, a_rows, p.a_mn_major);
                            prefetch_operand(&tmap_b, kb + p.l2_prefetch, c.n_blk * BN, BN,
                                             p.b_mn_major);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Let every copy this thread issued land before the CTA can exit
            // (immediate in normal operation: the MMA issuer consumed them all;
            // matters when some role gave up on a wait).
            {
                int s = stage;
                uint32_t ph = phase;
                const int pending = issued < STAGES ? issued : STAGES;
                for (int i = 0; i < pending; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        ph ^= 1u;
                    }
                    wait_phase_unwind(smem_addr(&ctl->full[s]), ph, 100000000ull);
                    // With multicast, also wait until every CTA of the cluster has
                    // released the slot, so no peer's commit arrives after exit.
                    if (p.mcast > 1) wait_phase_unwind(smem_addr(&ctl->empty[s]), ph, 100000000ull);
                }
            }
            (void)ok;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            bool ok = true;
            for (int32_t u = it.first; ok && u < p.num_units; u += it.stride) {
                const UnitCoord c = u == it.first ? c_first : unit_at(p, u);
                for (int32_t k0 = c.kb_begin; ok && k0 < c.kb_end; k0 += p.chunk_kb) {
                    const int32_t k1 = (k0 + p.chunk_kb < c.kb_end) ? k0 + p.chunk_kb : c.kb_end;
                    const uint32_t buf = acc_iter & 1u;
                    const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                    // (both accumulator buffers start free)
                    if (acc_iter >= 2 &&
                        !wait_phase(smem_addr(&ctl->tmem_empty[buf]), acc_phase ^ 1u, watch,
                                    kSiteMmaTmemEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    // (a slot never straddles chunks: chunk_kb is a multiple of KS)
                    for (int32_t kb = k0; kb < k1; kb += KS) {
                        const int32_t nsub = k1 - kb < KS ? k1 - kb : KS;
                        if (!wait_phase(smem_addr(&ctl->full[stage]), phase, watch, kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_step = desc_k_step(p.a_mn_major);
                        const uint32_t b_step = desc_k_step(p.b_mn_major);
#pragma unroll
                        for (int32_t j = 0; j < KS; ++j) {
                            if (j >= nsub) break;   // the slot's later k-blocks lie past the slice
                            const uint64_t a_desc = operand_desc<KS>(
                                ring + stage * L::kASlotBytes +
                                    kblock_offset(p.a_mn_major | p.a_half, kATileBytes, j),
                                p.a_mn_major);
                            const uint64_t b_desc = operand_desc<KS>(
                                ring_b + stage * L::kBTileBytes +
                                    kblock_offset(p.b_mn_major, L::kBSubBytes, j),
                                p.b_mn_major);
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k) {
                                umma_f16(d_tmem, a_desc + a_step * k, b_desc + b_step * k, p.idesc,
                                         (kb > k0 || j > 0 || k > 0) ? 1u : 0u);
                            }
                        }
                        if (p.mcast > 1)   // every CTA's copy of A in this slot is consumed
                            umma_commit_mcast(smem_addr(&ctl->empty[stage]),
                                              static_cast<uint16_t>((1u << p.mcast) - 1u));
                        else
                            umma_commit(smem_addr(&ctl->empty[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(smem_addr(&ctl->tmem_full[buf]));
                    ++acc_iter;
                }
            }
            // Drain: every MMA issued above completes before TMEM is released.
            umma_commit(smem_addr(&ctl->drain));
            wait_phase_unwind(smem_addr(&ctl->drain), 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;                    // TMEM lanes this warp may access
        const int row_in_tile = quad * 32 + lane;
        const int epi_tid = (warp - 2) * 32 + lane;   // 0..127
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        // This warp's two TMA-store buffers and which one is next.
        const uint32_t store_buf0 = staging + static_cast<uint32_t>((warp - 2) * 2 * L::kStoreBufBytes);
        // This warp's slot for a chunk's fused bias (after the control block).
        const uint32_t bias_slot = staging + static_cast<uint32_t>(L::kStagingBytes + L::kCtlBytes +
                                                                   (warp - 2) * kBiasSlotBytes);
        uint32_t store_sel = 0;
        uint32_t acc_iter = 0;
        bool ok = true;
        for (int32_t u = it.first; ok && u < p.num_units; u += it.stride) {
            const UnitCoord c = u == it.first ? c_first : unit_at(p, u);
            const int32_t row = c.m_blk * kBM + row_in_tile;
            const int32_t col0 = c.n_blk * BN;
            const bool split = p.split_k > 1 && !p.cluster_split;
            const bool cluster = p.cluster_split != 0;
            uint32_t* ws_row = nullptr;
            if (split)
                ws_row = reinterpret_cast<uint32_t*>(p.workspace) +
                         (static_cast<int64_t>(u) * kBM + row_in_tile) * BN;

            if constexpr (OUT == kOutI32) {
                uint32_t sum[BN];
#pragma unroll
                for (int i = 0; i < BN; ++i) sum[i] = 0u;
                for (int32_t k0 = c.kb_begin; k0 < c.kb_end; k0 += p.chunk_kb) {
                    const uint32_t buf = acc_iter & 1u;
                    const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                    if (!wait_phase(smem_addr(&ctl->tmem_full[buf]), acc_phase, watch,
                                    kSiteEpiTmemFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < BN / 32; ++j) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem_base + lane_addr + buf * BN + j * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            sum[j * 32 + i] +=
                                static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(&ctl->tmem_empty[buf]));
                    ++acc_iter;
                }
                if (!ok) break;
                // cluster split: park the sums behind the receive area of the ring
                // (idle now) until they are pushed after the cluster barrier
                if (cluster) fence_proxy_async_smem();
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    if (cluster) {
                        stage_row32<BN>(ring + SplitRecv<BN>::kBytes, row_in_tile, j * 32,
                                        &sum[j * 32]);
                    } else if (split) {
                        if (row < p.M) store_ws32(ws_row + j * 32, &sum[j * 32]);
                    } else if (p.direct_store) {
                        if (row < p.M) store_i32_row32(p.C, p.N, row, col0 + j * 32, &sum[j * 32]);
                    } else {
                        // 32 int32 columns = one 128-byte row of a store buffer.  A
                        // segment wholly outside C is skipped (warp-uniform), so every
                        // buffer switch matches one committed store group.
                        const int32_t y = c.m_blk * kBM + quad * 32;
                        const int32_t x = col0 + j * 32;
                        if (y < p.M && x < p.N) {
                            const uint32_t buf = store_buf0 + store_sel * L::kStoreBufBytes;
                            if (lane == 0) bulk_wait_group_read<1>();
                            __syncwarp();
                            stage_store_row(buf, lane, 0, &sum[j * 32], 8);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tmap_c, buf, x, y);
                                bulk_commit_group();
                            }
                            store_sel ^= 1u;
                        }
                    }
                }
            } else {
                const uint32_t buf = acc_iter & 1u;
                const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                // A fused bias / activation in the TMA-store path: the bias is staged
                // per chunk (bias_fetch2), the first chunk's fetched while the
                // accumulator is being computed.
                const bool epi = (p.bias != nullptr || p.act != 0) && !cluster && !split &&
                                 !p.direct_store;
                float2 b_next = make_float2(0.f, 0.f);
                if (epi) b_next = bias_fetch2(p.bias, p.N, col0 + 2 * lane);
                if (!wait_phase(smem_addr(&ctl->tmem_full[buf]), acc_phase, watch,
                                kSiteEpiTmemFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (cluster) {
                    // the accumulator stays in TMEM until it is pushed after the
                    // cluster barrier
                } else if (split || p.direct_store) {
#pragma unroll 1
                    for (int j = 0; j < BN / 32; ++j) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem_base + lane_addr + buf * BN + j * 32, v);
                        tmem_ld_wait();
                        if (row < p.M) {
                            if (split) {
                                store_ws32(ws_row + j * 32, v);
                            } else {
                                apply_bias_act<8>(v, p, col0 + j * 32);
                                store_half_row32<OUT>(p.C, p.N, row, col0 + j * 32, v);
                            }
                        }
                    }
                } else {
                    // 64 16-bit columns = one 128-byte store-buffer row per thread;
                    // segments wholly outside C are skipped (warp-uniform), so every
                    // buffer switch matches one committed store group.
                    const int32_t y = c.m_blk * kBM + quad * 32;
#pragma unroll 1
                    for (int sc = 0; sc < BN / 64; ++sc) {
                        const int32_t x = col0 + sc * 64;
                        if (y >= p.M || x >= p.N) continue;
                        const uint32_t sbuf = store_buf0 + store_sel * L::kStoreBufBytes;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                        if (epi) {
                            // (the warp's reads of the previous chunk's bias are done)
                            st_shared_f2(bias_slot + static_cast<uint32_t>(lane * 8), b_next);
                            __syncwarp();
                            if (sc + 1 < BN / 64) b_next = bias_fetch2(p.bias, p.N, x + 64 + 2 * lane);
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t v[32];
                            tmem_ld_32x32b_x32(tmem_base + lane_addr + buf * BN + sc * 64 + h * 32, v);
                            tmem_ld_wait();
                            if (epi)
                                apply_bias_act_staged<8>(v, p, bias_slot + static_cast<uint32_t>(h * 128));
                            uint32_t w[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[i] = pack2<OUT>(__uint_as_float(v[2 * i]),
                                                  __uint_as_float(v[2 * i + 1]));
                            stage_store_row(sbuf, lane, h * 4, w, 4);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmap_c, sbuf, x, y);
                            bulk_commit_group();
                        }
                        store_sel ^= 1u;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&ctl->tmem_empty[buf]));
                ++acc_iter;
            }

            if (split) {
                // Publish this slice; the last slice to arrive sums all slices in
                // slice order 0..S-1 (fixed order: identical results every run).
                // Rows beyond M are neither written nor read.
                __threadfence();
                named_bar_sync(1, kEpiWarps * 32);
                if (epi_tid == 0) {
                    const uint32_t prev = atomicAdd(&p.counters[c.tile], 1u);
                    const int32_t last = (prev == static_cast<uint32_t>(p.split_k - 1)) ? 1 : 0;
                    if (last) atomicExch(&p.counters[c.tile], 0u);
                    ctl->splitk_last = last;
                }
                named_bar_sync(1, kEpiWarps * 32);
                const int32_t last = *reinterpret_cast<volatile int32_t*>(&ctl->splitk_last);
                if (last && row < p.M) {
                    __threadfence();
                    const uint32_t* tile_ws = reinterpret_cast<const uint32_t*>(p.workspace) +
                                              (static_cast<int64_t>(c.tile) * p.split_k * kBM +
                                               row_in_tile) * BN;
                    const int64_t slice_stride = static_cast<int64_t>(kBM) * BN;
#pragma unroll 1
                    for (int j = 0; j < BN / 32; ++j) {
                        uint32_t v[32];
                        // integer mode keeps its BN int32 sums live: fewer loads in flight
                        reduce_slices32<OUT, (OUT == kOutI32 ? 2 : 4)>(tile_ws + j * 32,
                                                                       slice_stride, p.split_k, v);
                        if constexpr (OUT == kOutI32) {
                            store_i32_row32(p.C, p.N, row, col0 + j * 32, v);
                        } else {
                            apply_bias_act<8>(v, p, col0 + j * 32);
                            store_half_row32<OUT>(p.C, p.N, row, col0 + j * 32, v);
                        }
                    }
                }
            }
        }
        epi_ok = ok && it.first < p.num_units;
    }

    // ------------------------------------------- split-K reduction in the cluster
    if (p.cluster_split) {
        fence_proxy_async_smem();   // the TMA-written ring now receives peers' stores
        cluster_sync_all();         // every CTA's main loop is over: all rings are idle
        tc_fence_after();
        const UnitCoord c = unit_coord_fast(blockIdx.x, p);
        if (warp >= 2 && epi_ok) {
            // this warp's (idle) TMA-store buffers serve as its transpose staging
            const uint32_t stg = staging + static_cast<uint32_t>((warp - 2) * 2 * L::kStoreBufBytes);
            cluster_push_any<BN, OUT, 8>(p.split_k, ring, stg, tmem_base,
                                         ring + SplitRecv<BN>::kBytes, warp & 3, lane, c.split,
                                         1u, 0u);
        }
        cluster_sync_all();         // every slice has arrived at its owner
        if (warp >= 2)
            cluster_sum_store<BN, OUT, 8>(p, c.m_blk * kBM, c.n_blk * BN,
                                          static_cast<int>(cluster_ctarank()), ring,
                                          static_cast<int>(threadIdx.x) - 64);
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    if (p.mcast > 1)
        cluster_sync_all();   // no peer still sends copies or commits to this CTA
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    } else if (warp >= 2) {
        // This warp's bulk stores must have read their shared-memory source before
        // the CTA ends (while warp 1 frees TMEM); their global writes complete
        // with the grid.
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }
}

}  // namespace gbg
