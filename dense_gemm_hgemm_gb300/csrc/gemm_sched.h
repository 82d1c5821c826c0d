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

// Division by a run-time invariant d >= 1 as one multiply-high and a shift
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, section 4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, x / d = (mulhi(x, m) + x) >> l for every
// 0 <= x < 2^31 (mulhi(x, m) <= x, so the sum stays below 2^32).  A hardware
// integer divide is a long dependent chain on the GPU; tile coordinates are
// computed on the critical path of every kernel start.
struct FastDiv {
    uint32_t mul;
    uint32_t shift;
    int32_t d;
};

inline FastDiv make_fastdiv(int32_t d) {
    FastDiv f;
    f.d = d < 1 ? 1 : d;
    uint32_t l = 0;
    while ((uint64_t{1} << l) < static_cast<uint64_t>(f.d)) ++l;
    f.shift = l;
    f.mul = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - f.d)) / f.d + 1);
    return f;
}

GBG_HD int32_t fdiv(int32_t x, const FastDiv& f) {
#if defined(__CUDA_ARCH__)
    const uint32_t t = __umulhi(static_cast<uint32_t>(x), f.mul);
#else
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(static_cast<uint32_t>(x)) * f.mul) >> 32);
#endif
    return static_cast<int32_t>((t + static_cast<uint32_t>(x)) >> f.shift);
}

// Divisors of the raster order for `group` m-blocks per band over an n extent
// of n_ext: the band size, the group and the (partial) last band's height.
struct RasterDiv {
    FastDiv band, group, last;
};

inline RasterDiv make_raster_div(int32_t m_blocks, int32_t n_ext, int32_t group) {
    RasterDiv r;
    r.band = make_fastdiv(group * n_ext);
    r.group = make_fastdiv(group);
    r.last = make_fastdiv(m_blocks % group != 0 ? m_blocks % group : group);
    return r;
}

// raster_tile (below) with the divisions done by multiplication.
GBG_HD void raster_tile_fast(int32_t m_blocks, const RasterDiv& rd, int32_t tile, int32_t* m_blk,
                             int32_t* n_blk) {
    const int32_t g = fdiv(tile, rd.band);
    const int32_t r = tile - g * rd.band.d;
    const int32_t first_m = g * rd.group.d;
    const FastDiv& gs = (m_blocks - first_m < rd.group.d) ? rd.last : rd.group;
    const int32_t q = fdiv(r, gs);
    *m_blk = first_m + (r - q * gs.d);
    *n_blk = q;
}

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
