// gemm_config.h -- per-shape kernel configuration (host only).
//
// The pages tune tile shape, pipeline depth and swizzle with an RL agent
// ("H100 GEMM L2驻留优化：warp-specialized TMA异步拷贝与RL调优策略", paragraph on
// the RL agent and the "RL Search Space" list; "RL驱动CUDA L2 GEMM内核自动调优",
// paragraph on RL autotune).  Here the choice comes from a measured table
// (gemm_config_table.inc, written by tune.py from a sweep on the target GPU);
// shapes not in the table use the cost model below.
#pragma once
#include <stdint.h>

#include "gemm.h"
#include "gemm_launch.h"

namespace gbg {

struct TableEntry {
    int32_t M, N, K, dtype;
    int32_t block_n, split_k, raster_group, split_mode, cta_pair, direct_store, multicast,
        kblocks_per_stage;
};

#include "gemm_config_table.inc"   // static const TableEntry kTunedTable[]; kTunedCount

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Relative main-loop efficiency of a 128 x BN tile: per 64-wide k-block the MMA
// needs 128*BN*64/4096 cycles and shared memory delivers 128 B/cycle, so BN=256
// is MMA-bound, BN=128 sits at the shared-memory limit and BN=64 is
// shared-memory bound at about 2/3.
inline double tile_efficiency(int bn) { return bn == 256 ? 1.0 : (bn == 128 ? 0.9 : 0.6); }

inline gemm_config_t model_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int sms) {
    gemm_config_t c;
    c.stages = 0;
    c.max_ctas = 0;
    c.raster_group = 16;
    c.split_k = 1;
    c.split_mode = 0;
    c.cta_pair = 0;
    c.direct_store = 0;
    c.multicast = 0;
    c.l2_prefetch = 0;
    c.kblocks_per_stage = 0;
    const int64_t mb = ceil_div(M, kBM);
    const int64_t num_kb = ceil_div(K, kBK);
    const int cands_f[3] = {256, 128, 64};
    const int cands_i[2] = {128, 64};
    const int* cands = dtype == GEMM_I8_I32 ? cands_i : cands_f;
    const int ncand = dtype == GEMM_I8_I32 ? 2 : 3;
    double best = 1e300;
    c.block_n = cands[ncand - 1];
    for (int i = 0; i < ncand; ++i) {
        const int bn = cands[i];
        const int64_t tiles = mb * ceil_div(N, bn);
        const double waves = static_cast<double>(ceil_div(tiles, sms));
        const double t = waves * bn / tile_efficiency(bn);
        if (t < best * 0.999) {
            best = t;
            c.block_n = bn;
        }
    }
    // SM pairs (each SM streams half of B) once there is enough work per pair tile:
    // the measured table picks them exactly where (256 x 256 tiles) x K >= 2^17
    // (32 tiles from K = 4096, 64 from 2048, 128 from 1024, 256 from 512), with
    // 128-wide tiles while 256-wide ones would leave most pairs idle.
    const int64_t pair_tiles = ceil_div(M, 2 * kBM) * ceil_div(N, 256);
    if (mb >= 2 && pair_tiles * K >= (int64_t(1) << 17)) {
        c.block_n = pair_tiles * 5 >= sms * 2 ? 256 : 128;
        c.cta_pair = 1;
        c.raster_group = 8;
        return c;
    }
    // Few output tiles and a long K: one SM streams only ~110 GB/s, so slice K
    // over a cluster of 2/4/8 CTAs per tile (reduced in distributed shared memory),
    // at least four k-blocks per slice (the measured table splits from K = 1024).
    const int64_t tiles = mb * ceil_div(N, c.block_n);
    if (tiles * 2 <= sms && num_kb >= 16) {
        for (int s = 8; s >= 2; s /= 2) {
            const int64_t per = ceil_div(num_kb, s);
            if (tiles * s <= sms && num_kb >= 4 * s && ceil_div(num_kb, per) == s) {
                c.split_k = s;
                c.split_mode = 1;
                break;
            }
        }
    }
    return c;
}

inline gemm_config_t select_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype, int sms) {
    for (int i = 0; i < kTunedCount; ++i) {
        const TableEntry& e = kTunedTable[i];
        if (e.M == M && e.N == N && e.K == K && e.dtype == static_cast<int32_t>(dtype)) {
            gemm_config_t c;
            c.block_n = e.block_n;
            c.stages = 0;
            c.split_k = e.split_k;
            c.raster_group = e.raster_group;
            c.split_mode = e.split_mode;
            c.cta_pair = e.cta_pair;
            c.direct_store = e.direct_store;
            c.multicast = e.multicast;
            c.l2_prefetch = 0;
            c.kblocks_per_stage = e.kblocks_per_stage;
            c.max_ctas = 0;
            return c;
        }
    }
    return model_config(M, N, K, dtype, sms);
}

}  // namespace gbg
