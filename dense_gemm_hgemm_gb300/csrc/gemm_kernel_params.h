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
};

}  // namespace gbg
