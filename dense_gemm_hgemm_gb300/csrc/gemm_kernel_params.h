// gemm_kernel_params.h -- kernel parameter block and constants shared by the
// kernels and the host planner.
#pragma once
#include <stdint.h>

#include "gemm_sched.h"

namespace gbg {

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kATileBytes = kBM * kBK * 2;   // 16 KiB

enum OutKind : int { kOutF16 = 0, kOutBF16 = 1, kOutI32 = 2 };

// Compiled forms of a kernel.  General: every mode is a run-time field of
// KParams.  Plain: one K slice, no multicast, TMA stores, K-contiguous operands,
// no L2 prefetch distance, no fused bias or activation.  Cluster split (one-SM
// kernel): as plain, but the K slices of a tile form one thread-block cluster
// (split_k stays a run-time value).  Epilogue: as plain, with the fused bias and
// activation run-time values (what a plain plan launches for such a call).  The
// fixed fields become constants, so the code of the other modes compiles out of
// the launch's critical path.
enum KernelForm : int { kFormGeneral = 0, kFormPlain = 1, kFormClusterSplit = 2, kFormEpilogue = 3 };

// Forms whose copy thread arms the ring's first slots before the dependency
// wait.  (The general and epilogue forms arm each slot in their loop: the extra
// copy-issue code measured slower next to a fused epilogue.)
template <int FORM>
inline constexpr bool kArmedCopy = FORM == kFormPlain || FORM == kFormClusterSplit;

// Shared memory per epilogue warp for the fused bias of one 64-column chunk.
constexpr int kBiasSlotBytes = 64 * 4;

// SM-pair integer tiles wider than 128 columns keep their int32 sums in registers
// across eight epilogue warps (two per TMEM lane quarter, splitting the columns).
template <int BN, int OUT>
inline constexpr int kPairEpiWarps = OUT == kOutI32 && BN > 128 ? 8 : kEpiWarps;
// Threads of an SM-pair CTA (host side): producer and MMA warps + epilogue warps.
constexpr int pair_threads(int bn, int out) { return 64 + 32 * (out == kOutI32 && bn > 128 ? 8 : kEpiWarps); }

// Wait-site codes written to the error word when a wait runs out.
enum WaitSite : int32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteEpiTmemFull = 4,
};

struct KParams {
    int32_t M, N, K;
    int32_t num_kb;         // ceil(K / kBK)
    int32_t m_blocks, n_blocks;
    int32_t split_k;        // K slices per tile
    int32_t cluster_split;  // 1: the split_k slices of a tile form one thread-block
                            // cluster and are reduced through distributed shared
                            // memory (one unit per CTA); 0: workspace + last arriver
    int32_t kb_per_split;   // k-blocks per slice
    int32_t chunk_kb;       // k-blocks per accumulation chunk (integer mode), else >= kb_per_split
    int32_t raster_group;
    int32_t direct_store;   // 1: epilogue stores C with 16-byte st.global per thread; 0: TMA stores
    int32_t a_mn_major;     // 1: A stored K x M (M contiguous); 0: M x K (K contiguous)
    int32_t b_mn_major;     // 1: B stored K x N (N contiguous); 0: N x K (K contiguous)
    int32_t mcast;          // > 1: clusters of mcast CTAs own mcast adjacent N-tiles of the same
                            // rows; each loads 1/mcast of the A tile and multicasts it to all
                            // (num_units then counts tile groups)
    int32_t l2_prefetch;    // > 0: the producer also prefetches k-block kb + l2_prefetch into L2
    int32_t a_half;         // 1 (M <= 64, one-SM kernel): only A rows 0..63 of the tile are
                            // copied, 8 KiB per k-block (k-block j of a slot at 8 KiB * j); the
                            // MMA's rows 64..127 read whatever the slot holds and are never stored
    int32_t num_units;      // m_blocks * n_blocks * split_k
    uint32_t idesc;         // tcgen05 instruction descriptor
    uint32_t tx_extra;      // extra bytes each ring slot expects (0 in normal operation)
    const float* bias;      // per-column bias (N fp32 values) or null
    int32_t act;            // 0 none, 1 ReLU, 2 GELU (erf), 3 SiLU: C = act(A B^T + bias)
    void* C;
    void* workspace;        // split-K partials: [num_units][kBM][BN] fp32 (int32 in integer mode)
    uint32_t* counters;     // split-K arrival counter per tile (self-resetting)
    int32_t* error_word;
    uint64_t timeout_ns;
    // Multiply-shift divisors of the work decomposition (see FastDiv): by
    // split_k, and of the raster over (m_blocks, raster_n) in bands of
    // raster_group, where raster_n is n_blocks, or the number of n-block groups
    // with multicast (mcast = 1 << mcast_shift).
    FastDiv fd_split;
    RasterDiv rd;
    int32_t raster_n;
    int32_t mcast_shift;
};

// Coordinates of unit u (as unit_coord) from the plan's precomputed divisors.
GBG_HD UnitCoord unit_coord_fast(int32_t u, const KParams& p) {
    UnitCoord c;
    c.tile = fdiv(u, p.fd_split);
    c.split = u - c.tile * p.split_k;
    raster_tile_fast(p.m_blocks, p.rd, c.tile, &c.m_blk, &c.n_blk);
    c.kb_begin = c.split * p.kb_per_split;
    const int32_t e = c.kb_begin + p.kb_per_split;
    c.kb_end = e < p.num_kb ? e : p.num_kb;
    return c;
}

// Fill the divisor fields from the plain ones (m_blocks, n_blocks, split_k,
// raster_group, mcast).
inline void set_divisors(KParams* p) {
    p->fd_split = make_fastdiv(p->split_k);
    const int32_t mc = p->mcast > 1 ? p->mcast : 1;
    p->raster_n = (p->n_blocks + mc - 1) / mc;
    int32_t sh = 0;
    while ((1 << sh) < mc) ++sh;
    p->mcast_shift = sh;
    const int32_t g = p->raster_group < 1 ? 1 : p->raster_group;
    p->rd = make_raster_div(p->m_blocks, p->raster_n, g);
}

}  // namespace gbg
