// gemm_sched.h -- work decomposition shared by the host planner and the kernels.
//
// Output tiles are kBM x BN.  A "unit" is one (tile, K-slice) pair; with
// split-K = S a tile owns S consecutive units.  A persistent CTA b processes
// units b, b + gridDim.x, b + 2*gridDim.x, ...
//
// Tile order ("raster"): linear tile ids run over bands of `group` m-blocks;
// inside a band the m-block index moves fastest, so the CTAs that run at the
// same time cover a compact group x (ctas/group) block of C and share the A and
// B panels they stream through L2.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define GBG_HD __host__ __device__ __forceinline__
#else
#define GBG_HD inline
#endif

namespace gbg {

constexpr int kBM = 128;   // tile rows = tcgen05 M (one TMEM lane per row)
constexpr int kBK = 64;    // K elements per pipeline stage (128 bytes of fp16/bf16)

GBG_HD void raster_tile(int32_t m_blocks, int32_t n_blocks, int32_t group, int32_t tile,
                        int32_t* m_blk, int32_t* n_blk) {
    const int32_t band = group * n_blocks;
    const int32_t g = tile / band;
    const int32_t r = tile - g * band;
    const int32_t first_m = g * group;
    const int32_t rem = m_blocks - first_m;
    const int32_t gsize = rem < group ? rem : group;
    *m_blk = first_m + r % gsize;
    *n_blk = r / gsize;
}

struct UnitCoord {
    int32_t tile;      // linear tile id (index of the split-K counter)
    int32_t m_blk, n_blk;
    int32_t split;     // K-slice index
    int32_t kb_begin, kb_end;   // k-block range [begin, end)
};

GBG_HD UnitCoord unit_coord(int32_t unit, int32_t split_k, int32_t kb_per_split, int32_t num_kb,
                            int32_t m_blocks, int32_t n_blocks, int32_t group) {
    UnitCoord c;
    c.tile = unit / split_k;
    c.split = unit - c.tile * split_k;
    raster_tile(m_blocks, n_blocks, group, c.tile, &c.m_blk, &c.n_blk);
    c.kb_begin = c.split * kb_per_split;
    const int32_t e = c.kb_begin + kb_per_split;
    c.kb_end = e < num_kb ? e : num_kb;
    return c;
}

}  // namespace gbg
