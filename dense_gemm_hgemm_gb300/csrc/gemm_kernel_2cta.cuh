// gemm_kernel_2cta.cuh -- the SM-pair (tcgen05 cta_group::2) variant of the TN GEMM.
//
// A thread-block cluster of two CTAs (ranks 0 = leader, 1 = peer, on two SMs)
// computes a 256 x BN output tile (BN = 128, 224 or 256):
//   * each CTA streams its own 128 rows of A (128 x 64 per stage) and its half
//     of the tile's B rows (BN/2 x 64 per stage) into its own 128B-swizzled
//     ring; both CTAs' copies count bytes on the LEADER's `full` barrier;
//   * one thread of the leader issues tcgen05.mma.cta_group::2 (M=256, N=BN,
//     K=16): the hardware reads A and B from both CTAs' shared memory and
//     writes accumulator rows 0-127 to the leader's TMEM, rows 128-255 to the
//     peer's; tcgen05.commit multicasts ring-slot releases and "accumulator
//     ready" to the same barriers in both CTAs;
//   * each CTA's four epilogue warps drain its own TMEM half and TMA-store it
//     (64 columns per store; the last 32 columns of a 224-wide tile are stored
//     from registers, as a 64-column box would reach into the next tile), then
//     arrive (locally or remotely) on the leader's `tmem_empty` barrier.
// Per SM this moves 32 KiB per 64-wide k-block for 128 x BN x 64 MACs (BN=256)
// instead of 48 KiB in the one-SM kernel, and the ring holds 6 stages.
//
// Same conventions as gemm_kernel.cuh: persistent over tiles (one cluster per SM
// pair), double-buffered TMEM accumulator, bounded waits with an error word,
// programmatic dependent launch, L2 prefetch before the dependency wait.
//
// A multicast (mcast = 2): a cluster of four CTAs holds two pairs that compute
// adjacent N-tiles (2g, 2g+1) of the same 256 rows.  CTA (pair q, half h) loads
// rows [64q, 64q+64) of its half's 128 A rows and multicasts them to CTA (0, h)
// and CTA (1, h), so each A row crosses from L2 once for both pairs.  Each pair
// leader's MMA commit releases the slot in all four CTAs (every empty barrier
// counts both pairs), so a slot is refilled only when both pairs consumed it; a
// tile past N loads zeros and stores nothing.
//
// Split-K in the cluster (cluster_split, S = 2 or 4): a cluster of 2S CTAs holds
// S pairs (ranks 2s, 2s+1 form pair s) that compute K-slices s of one 256 x BN
// tile; each CTA stages its fp32 partial rows in its (then idle) ring, and CTA
// (s, half h) sums rows [s*128/S, (s+1)*128/S) of half h over the S pairs in
// slice order through distributed shared memory.
#pragma once

#include "gemm_kernel.cuh"

namespace gbg {

// KS = 64-wide k-blocks per ring slot (2 or 4: each operand's KS k-blocks in one
// 3-D copy, as in the one-SM kernel).
template <int BN, int STAGES, int KS = 1>
struct SmemLayout2 {
    static constexpr int kBSubBytes = (BN / 2) * kBK * 2;    // this CTA's half of B, one k-block
    static constexpr int kASlotBytes = KS * kATileBytes;
    static constexpr int kBTileBytes = KS * kBSubBytes;
    static constexpr int kStageBytes = kASlotBytes + kBTileBytes;
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kStoreBufBytes = 32 * 128;
    static constexpr int kStagingBytes = kEpiWarps * 2 * kStoreBufBytes;
    static constexpr int kCtlBytes = 256;
    static constexpr int kBiasBytes = kEpiWarps * kBiasSlotBytes;   // after the control block
    static constexpr int kTotal = 1024 + kRingBytes + kStagingBytes + kCtlBytes + kBiasBytes;
    static_assert(kBTileBytes % 1024 == 0, "128B-swizzle tiles must stay 1024-byte aligned");
    static_assert(kTotal <= 232448, "exceeds the 227 KiB a CTA may use");
};

// Wait-site code for a TMEM address mismatch between the two CTAs of a pair.
constexpr int32_t kSitePairTmem = 5;

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T, M=256, N=BN, K=16.
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at this shared-memory offset in every CTA of
// `cta_mask` when all prior tcgen05.mma of this thread are done.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// TMA load into this CTA's shared memory whose bytes are counted on a barrier
// that may live in the peer CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

// Multicast form: the box lands at the same shared-memory offset in every CTA of
// `cta_mask`, and for each destination CTA the bytes are counted on the barrier
// at `bar_cluster`'s offset in that destination's pair leader (checked on GB300:
// with the barrier operand naming the issuing pair's leader, destinations 0/2
// and 1/3 of a four-CTA cluster all complete the barriers of CTAs 0 and 2).
__device__ __forceinline__ void tma_load_2d_pair_mcast(uint32_t dst, const CUtensorMap* map,
                                                       uint32_t bar_cluster, int32_t x, int32_t y,
                                                       uint16_t cta_mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "h"(cta_mask)
        : "memory");
}

// 3-D form (operand map viewed as 64 elements x rows x k-blocks).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// load_operand_kb for the pair kernel (bytes counted on the leader's barrier).
template <int KS>
__device__ __forceinline__ void load_operand_kb_pair(uint32_t dst, const CUtensorMap* map,
                                                     uint32_t bar_cluster, int32_t kb, int32_t row0,
                                                     int32_t rows, int32_t mn_major) {
    if (!mn_major) {
        tma_load_3d_pair(dst, map, bar_cluster, 0, row0, kb);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i)
        tma_load_2d_pair(dst + static_cast<uint32_t>(i * KS) * 8192u, map, bar_cluster,
                         row0 + i * 64, kb * kBK);
}

// load_operand for the pair kernel (bytes counted on the leader's barrier).
__device__ __forceinline__ void load_operand_pair(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar_cluster, int32_t kb, int32_t row0,
                                                  int32_t rows, int32_t mn_major) {
    if (!mn_major) {
        tma_load_2d_pair(dst, map, bar_cluster, kb * kBK, row0);
        return;
    }
    for (int32_t i = 0; i < rows / 64; ++i)
        tma_load_2d_pair(dst + static_cast<uint32_t>(i) * 8192u, map, bar_cluster, row0 + i * 64,
                         kb * kBK);
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "n"(kWaitHintNs)
        : "memory");
    return done != 0;
}

// As wait_phase, with cluster-scope acquire (the arrivals come from both CTAs).
__device__ __forceinline__ bool wait_phase_cluster(uint32_t bar, uint32_t parity, const Watch& w,
                                                   int32_t site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
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

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// FORM: kFormGeneral, kFormPlain or kFormEpilogue (see KernelForm; the host picks it).
template <int BN, int STAGES, int OUT, int KS = 1, int FORM = kFormGeneral>
__global__ void __launch_bounds__(64 + 32 * kPairEpiWarps<BN, OUT>, 1)
    gemm_tn_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_c, const KParams p_in) {
    static_assert(FORM == kFormGeneral || FORM == kFormPlain || FORM == kFormEpilogue,
                  "SM-pair kernel forms");
    const KParams p = form_params<FORM>(p_in);
    using L = SmemLayout2<BN, STAGES, KS>;
    static_assert(KS == 1 || KS == 2 || KS == 4, "k-blocks per ring slot");
    // integer tiles wider than 128: eight epilogue warps, one store buffer each
    constexpr bool kIntWide = OUT == kOutI32 && BN > 128;
    constexpr int kEpi = kPairEpiWarps<BN, OUT>;
    static_assert(((OUT == kOutI32 && !kIntWide) ? 2 : 1) * SplitRecv<BN>::kBytes <= L::kRingBytes,
                  "split-K receive area (and parked integer sums) must fit in the ring");
    static_assert(BN == 128 || BN == 224 || BN == 256, "pair tile width");
    static_assert(kEpi * (kIntWide ? 1 : 2) * L::kStoreBufBytes <= L::kStagingBytes,
                  "epilogue store buffers");
    // two accumulator buffers of BN columns; an allocation is a power of two
    constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256u : 512u;
    constexpr uint32_t kPairTx = 2 * L::kStageBytes;   // both CTAs' bytes per stage

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t ring = smem_addr(smem);
    const uint32_t ring_b = ring + STAGES * L::kASlotBytes;
    const uint32_t staging = ring + L::kRingBytes;
    SharedCtl<STAGES>* ctl =
        reinterpret_cast<SharedCtl<STAGES>*>(smem + L::kRingBytes + L::kStagingBytes);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1u;                  // 0: leader, 1: peer (within the pair)
    const uint32_t lead = crank & ~1u;                 // cluster rank of this pair's leader
    const uint16_t pair_mask = static_cast<uint16_t>(3u << lead);
    const bool leader = rank == 0;
    // With A multicast a unit is a group of two n-tiles owned by one four-CTA
    // cluster; otherwise one tile (or K-slice) per pair.
    const bool mcast = p.mcast > 1;
    const uint32_t qpair = (crank >> 1) & 1u;          // pair within a multicast cluster
    const uint16_t release_mask = mcast ? static_cast<uint16_t>(0xFu) : pair_mask;
    const uint16_t a_mask = static_cast<uint16_t>((1u << rank) | (1u << (2u + rank)));
    const int32_t pair = static_cast<int32_t>(blockIdx.x >> (mcast ? 2 : 1));
    const int32_t npairs = static_cast<int32_t>(gridDim.x >> (mcast ? 2 : 1));
    auto coord = [&](int32_t u) {
        UnitCoord c = unit_coord_fast(u, p);
        if (mcast) c.n_blk = c.n_blk * 2 + static_cast<int32_t>(qpair);
        return c;
    };

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        prefetch_tmap(&tmap_c);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), mcast ? 2 : 1);   // both pairs' releases
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&ctl->tmem_full[b]), 1);
            mbar_init(smem_addr(&ctl->tmem_empty[b]), 2 * kEpi);   // both CTAs' epilogues
        }
        mbar_init(smem_addr(&ctl->drain), 1);
        ctl->abort = 0;
        ctl->splitk_last = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const Watch watch{&ctl->abort, p.error_word, p.timeout_ns};
    if (!leader && threadIdx.x == 0) {
        // The leader's MMAs address the peer's TMEM with the leader's address.
        const uint32_t lead_base = ld_dsmem_u32(map_to_rank(smem_addr(&ctl->tmem_base), lead));
        if (lead_base != tmem_base) {
            atomicCAS(p.error_word, 0, kSitePairTmem);
            ctl->abort = 1;
        }
    }

    bool epi_ok = false;   // epilogue: this CTA's accumulator is complete (split-K in the cluster)
    // This pair's first unit, worked out while the previous kernel may still run.
    const UnitCoord c_first = coord(pair);
    // Plain form: ring slots of the first unit that the leader's copy thread arms
    // before the wait (shared memory only), so that right after it both copy
    // threads only issue their copies (kArmedCopy).
    int32_t n_armed = 0;
    if constexpr (kArmedCopy<FORM>) {
        if (warp == 0 && lane == 0 && pair < p.num_units) {
            const int32_t nslots = (c_first.kb_end - c_first.kb_begin + KS - 1) / KS;
            n_armed = nslots < STAGES ? nslots : STAGES;
            if (leader)
                for (int32_t s = 0; s < n_armed; ++s)
                    mbar_arrive_expect_tx(smem_addr(&ctl->full[s]), kPairTx + p.tx_extra);
        }
    }
    if (warp == 0 && lane == 0 && pair < p.num_units) {
        const UnitCoord c = c_first;
        const int32_t ahead = STAGES * KS > p.l2_prefetch ? STAGES * KS : p.l2_prefetch;
        const int32_t kb_end = c.kb_begin + ahead < c.kb_end ? c.kb_begin + ahead : c.kb_end;
        // with multicast, this CTA's 64-row share of its half's A rows
        const int32_t a_rows = mcast ? kBM / 2 : kBM;
        const int32_t a_row = c.m_blk * 2 * kBM + static_cast<int32_t>(rank) * kBM +
                              (mcast ? static_cast<int32_t>(qpair) * a_rows : 0);
        const int32_t b_row = c.n_blk * BN + static_cast<int32_t>(rank) * (BN / 2);
        for (int32_t kb = c.kb_begin; kb < kb_end; kb += KS) {
            if constexpr (KS > 1) {
                prefetch_operand_kb(&tmap_a, kb, a_row, a_rows, p.a_mn_major);
                prefetch_operand_kb(&tmap_b, kb, b_row, BN / 2, p.b_mn_major);
            } else {
                prefetch_operand(&tmap_a, kb, a_row, a_rows, p.a_mn_major);
                prefetch_operand(&tmap_b, kb, b_row, BN / 2, p.b_mn_major);
            }
        }
    }
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if constexpr (kArmedCopy<FORM>) {
            // (no multicast, no L2 prefetch distance, K-contiguous operands)
            if (lane == 0) {   // the thread that armed the first slots
                auto issue = [&](int stage, int32_t kb, const UnitCoord& c) {
                    const int32_t a_row = c.m_blk * 2 * kBM + static_cast<int32_t>(rank) * kBM;
                    const int32_t b_row = c.n_blk * BN + static_cast<int32_t>(rank) * (BN / 2);
                    const uint32_t full_lead = map_to_rank(smem_addr(&ctl->full[stage]), lead);
                    if constexpr (KS > 1) {
                        load_operand_kb_pair<KS>(ring + stage * L::kASlotBytes, &tmap_a, full_lead,
                                                 kb, a_row, kBM, 0);
                        load_operand_kb_pair<KS>(ring_b + stage * L::kBTileBytes, &tmap_b,
                                                 full_lead, kb, b_row, BN / 2, 0);
                    } else {
                        load_operand_pair(ring + stage * kATileBytes, &tmap_a, full_lead, kb,
                                          a_row, kBM, 0);
                        load_operand_pair(ring_b + stage * L::kBTileBytes, &tmap_b, full_lead, kb,
                                          b_row, BN / 2, 0);
                    }
                };
                for (int32_t s = 0; s < n_armed; ++s) issue(s, c_first.kb_begin + s * KS, c_first);
                int stage = n_armed == STAGES ? 0 : n_armed;
                uint32_t phase = n_armed == STAGES ? 1u : 0u;
                int issued = n_armed;
                bool ok = true;
                for (int32_t u = pair; ok && u < p.num_units; u += npairs) {
                    const UnitCoord c = u == pair ? c_first : coord(u);
                    for (int32_t kb = u == pair ? c.kb_begin + n_armed * KS : c.kb_begin;
                         kb < c.kb_end; kb += KS) {
                        if (issued >= STAGES &&
                            !wait_phase(smem_addr(&ctl->empty[stage]), phase ^ 1u, watch,
                                        kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        if (leader)
                            mbar_arrive_expect_tx(smem_addr(&ctl->full[stage]), kPairTx + p.tx_extra);
                        issue(stage, kb, c);
                        ++issued;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                // both CTAs' copies count on the leader's barriers: they land before
                // the pair can leave (see below)
                const int pending = issued < STAGES ? issued : STAGES;
                for (int i = 0; i < pending; ++i) {
                    if (--stage < 0) {
                        stage = STAGES - 1;
                        phase ^= 1u;
                    }
                    if (leader) wait_phase_unwind(smem_addr(&ctl->full[stage]), phase, 100000000ull);
                }
            }
        } else if (elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int32_t u = pair; ok && u < p.num_units; u += npairs) {
                const UnitCoord c = u == pair ? c_first : coord(u);
                const int32_t a_row = c.m_blk * 2 * kBM + static_cast<int32_t>(rank) * kBM;
                const int32_t b_row = c.n_blk * BN + static_cast<int32_t>(rank) * (BN / 2);
                for (int32_t kb = c.kb_begin; kb < c.kb_end; kb += KS) {
                    // (the first pass over the ring finds every slot free)
                    if (issued >= STAGES &&
                        !wait_phase(smem_addr(&ctl->empty[stage]), phase ^ 1u, watch,
                                    kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_local = smem_addr(&ctl->full[stage]);
                    if (leader) mbar_arrive_expect_tx(full_local, kPairTx + p.tx_extra);
                    const uint32_t full_lead = map_to_rank(full_local, lead);
                    if constexpr (KS > 1) {
                        // the slot's KS k-blocks of each operand in one copy (full box always)
                        load_operand_kb_pair<KS>(ring + stage * L::kASlotBytes, &tmap_a, full_lead,
                                                 kb, a_row, kBM, p.a_mn_major);
                        load_operand_kb_pair<KS>(ring_b + stage * L::kBTileBytes, &tmap_b, full_lead,
                                                 kb, b_row, BN / 2, p.b_mn_major);
                        if (p.l2_prefetch > 0 && kb + p.l2_prefetch < c.kb_end) {
                            prefetch_operand_kb(&tmap_a, kb + p.l2_prefetch, a_row, kBM, p.a_mn_major);
                            prefetch_operand_kb(&tmap_b, kb + p.l2_prefetch, b_row, BN / 2,
                                                p.b_mn_major);
                        }
                    } else {
                        if (mcast) {
                            // this CTA's 64 rows of its half's A tile, into the same slot
                            // offset of the matching CTA of both pairs; the bytes count on
                            // each destination pair's leader barrier (K-major: 64 rows of
                            // 128 B; M-major: one 64-element block, either way 8 KiB in)
                            const uint32_t a_dst = ring + stage * kATileBytes + qpair * 8192u;
                            const int32_t a_r = a_row + static_cast<int32_t>(qpair) * (kBM / 2);
                            if (p.a_mn_major)
                                tma_load_2d_pair_mcast(a_dst, &tmap_a, full_lead, a_r, kb * kBK, a_mask);
                            else
                                tma_load_2d_pair_mcast(a_dst, &tmap_a, full_lead, kb * kBK, a_r, a_mask);
                        } else {
                            load_operand_pair(ring + stage * kATileBytes, &tmap_a, full_lead, kb,
                                              a_row, kBM, p.a_mn_major);
                        }
                        load_operand_pair(ring_b + stage * L::kBTileBytes, &tmap_b, full_lead, kb,
                                          b_row, BN / 2, p.b_mn_major);
                        if (p.l2_prefetch > 0 && kb + p.l2_prefetch < c.kb_end) {
                            if (mcast)
                                prefetch_operand(&tmap_a, kb + p.l2_prefetch,
                                                 a_row + static_cast<int32_t>(qpair) * (kBM / 2),
                                                 kBM / 2, p.a_mn_major);
                            else
                                prefetch_operand(&tmap_a, kb + p.l2_prefetch, a_row, kBM,
                                                 p.a_mn_major);
                            prefetch_operand(&tmap_b, kb + p.l2_prefetch, b_row, BN / 2,
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
            {
                // Both CTAs' copies count on the leader's barriers: wait for them to
                // land before the pair can leave (immediate in normal operation).
                // With multicast every CTA also waits until both pairs have released
                // its last slots, so no peer's commit arrives after it exits.
                int s = stage;
                uint32_t ph = phase;
                const int pending = issued < STAGES ? issued : STAGES;
                for (int i = 0; i < pending; ++i) {
                    if (--s < 0) {
                        s = STAGES - 1;
                        ph ^= 1u;
                    }
                    if (leader) wait_phase_unwind(smem_addr(&ctl->full[s]), ph, 100000000ull);
                    if (mcast) wait_phase_unwind(smem_addr(&ctl->empty[s]), ph, 100000000ull);
                }
            }
            (void)ok;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (leader && elect_one_sync()) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_iter = 0;
            bool ok = true;
            for (int32_t u = pair; ok && u < p.num_units; u += npairs) {
                const UnitCoord c = u == pair ? c_first : coord(u);
                // One accumulation per chunk of k-blocks (the whole K range except in
                // integer mode, where a chunk keeps every fp32 partial sum exact).
                for (int32_t k0 = c.kb_begin; ok && k0 < c.kb_end; k0 += p.chunk_kb) {
                    const int32_t k1 = (k0 + p.chunk_kb < c.kb_end) ? k0 + p.chunk_kb : c.kb_end;
                    const uint32_t buf = acc_iter & 1u;
                    const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                    // (both accumulator buffers start free)
                    if (acc_iter >= 2 &&
                        !wait_phase_cluster(smem_addr(&ctl->tmem_empty[buf]), acc_phase ^ 1u,
                                            watch, kSiteMmaTmemEmpty)) {
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
                                ring + stage * L::kASlotBytes + kblock_offset(p.a_mn_major, kATileBytes, j),
                                p.a_mn_major);
                            const uint64_t b_desc = operand_desc<KS>(
                                ring_b + stage * L::kBTileBytes +
                                    kblock_offset(p.b_mn_major, L::kBSubBytes, j),
                                p.b_mn_major);
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k)
                                umma_f16_pair(d_tmem, a_desc + a_step * k, b_desc + b_step * k,
                                              p.idesc, (kb > k0 || j > 0 || k > 0) ? 1u : 0u);
                        }
                        umma_commit_pair(smem_addr(&ctl->empty[stage]), release_mask);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair(smem_addr(&ctl->tmem_full[buf]), pair_mask);
                    ++acc_iter;
                }
            }
            umma_commit_pair(smem_addr(&ctl->drain), static_cast<uint16_t>(1u << lead));
            wait_phase_unwind(smem_addr(&ctl->drain), 0, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quad = warp & 3;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t store_buf0 =
            staging + static_cast<uint32_t>((warp - 2) * (kIntWide ? 1 : 2) * L::kStoreBufBytes);
        uint32_t store_sel = 0;
        uint32_t acc_iter = 0;
        bool ok = true;
        for (int32_t u = pair; ok && u < p.num_units; u += npairs) {
            const UnitCoord c = u == pair ? c_first : coord(u);
            const int32_t y = c.m_blk * 2 * kBM + static_cast<int32_t>(rank) * kBM + quad * 32;
            const int32_t col0 = c.n_blk * BN;
            const int row_in_tile = quad * 32 + lane;
            if constexpr (kIntWide) {
                // Integer mode, 224/256-wide tiles: two warps per TMEM lane quarter;
                // warps 2-5 take columns [0, 128) of their 32 rows, warps 6-9 columns
                // [128, BN).  Each exact fp32 chunk is rounded to int32 and added in
                // registers (mod 2^32); the sums are stored once per tile.
                const int c_lo = ((warp - 2) >> 2) * 128;
                const int nj = c_lo == 0 ? 4 : (BN - 128) / 32;
                uint32_t sum[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) sum[i] = 0u;
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
                    for (int j = 0; j < 4; ++j) {
                        if (j >= nj) break;   // warp-uniform
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem_base + lane_addr + buf * BN + c_lo + j * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            sum[j * 32 + i] +=
                                static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[i])));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_remote(map_to_rank(smem_addr(&ctl->tmem_empty[buf]), lead));
                    ++acc_iter;
                }
                if (!ok) break;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int32_t x = col0 + c_lo + j * 32;   // 32 int32 = one buffer row
                    if (j >= nj || y >= p.M || x >= p.N) continue;   // warp-uniform
                    if (lane == 0) bulk_wait_group_read<0>();   // one buffer per warp
                    __syncwarp();
                    stage_store_row(store_buf0, lane, 0, &sum[j * 32], 8);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_c, store_buf0, x, y);
                        bulk_commit_group();
                    }
                }
                continue;
            } else if constexpr (OUT == kOutI32) {
                // Integer mode: round each exact fp32 chunk to int32 and add (mod 2^32).
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
                    if (lane == 0)
                        mbar_arrive_remote(map_to_rank(smem_addr(&ctl->tmem_empty[buf]), lead));
                    ++acc_iter;
                }
                if (!ok) break;
                if (p.cluster_split) {
                    // park the sums behind the receive area of the (idle) ring until
                    // they are pushed after the cluster barrier
                    fence_proxy_async_smem();
#pragma unroll
                    for (int j = 0; j < BN / 32; ++j)
                        stage_row32<BN>(ring + SplitRecv<BN>::kBytes, row_in_tile, j * 32,
                                        &sum[j * 32]);
                    continue;
                }
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    const int32_t x = col0 + j * 32;   // 32 int32 = one 128-byte buffer row
                    if (y >= p.M || x >= p.N) continue;   // warp-uniform
                    const uint32_t sbuf = store_buf0 + store_sel * L::kStoreBufBytes;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    stage_store_row(sbuf, lane, 0, &sum[j * 32], 8);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_c, sbuf, x, y);
                        bulk_commit_group();
                    }
                    store_sel ^= 1u;
                }
                continue;
            }
            const uint32_t buf = acc_iter & 1u;
            const uint32_t acc_phase = (acc_iter >> 1) & 1u;
            // A fused bias / activation: the bias is staged per chunk in this warp's
            // slot (see the one-SM kernel), the first chunk's fetched while the
            // accumulator is being computed.
            const bool epi = (p.bias != nullptr || p.act != 0) && !p.cluster_split;
            const uint32_t bias_slot =
                staging + static_cast<uint32_t>(L::kStagingBytes + L::kCtlBytes +
                                                (warp - 2) * kBiasSlotBytes);
            float2 b_next = make_float2(0.f, 0.f);
            if (epi) b_next = bias_fetch2(p.bias, p.N, col0 + 2 * lane);
            if (!wait_phase(smem_addr(&ctl->tmem_full[buf]), acc_phase, watch, kSiteEpiTmemFull)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // (cluster split: the accumulator stays in TMEM until it is pushed after
            // the cluster barrier)
#pragma unroll 1
            for (int sc = 0; sc < BN / 64; ++sc) {
                const int32_t x = col0 + sc * 64;
                if (p.cluster_split || y >= p.M || x >= p.N) continue;   // warp-uniform
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
                    if (epi) apply_bias_act_staged<8>(v, p, bias_slot + static_cast<uint32_t>(h * 128));
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack2<OUT>(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
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
            if constexpr (BN % 64 != 0) {
                // The tile's last 32 columns (BN = 224): a 64-column store box would
                // reach into the next tile, so each thread stores its own row.
                const int32_t x = col0 + (BN / 64) * 64;
                if (!p.cluster_split && y < p.M && x < p.N) {   // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + lane_addr + buf * BN + (BN / 64) * 64, v);
                    tmem_ld_wait();
                    apply_bias_act<8>(v, p, x);
                    if (y + lane < p.M) store_half_row32<OUT>(p.C, p.N, y + lane, x, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = smem_addr(&ctl->tmem_empty[buf]);
                mbar_arrive_remote(map_to_rank(bar, lead));
            }
            ++acc_iter;
        }
        epi_ok = ok && pair < p.num_units;
    }

    // ------------------------------------- split-K reduction across the cluster's pairs
    // (tile widths that are multiples of 64, integer ones of 128: the host splits no
    // other tile)
    if constexpr (BN % 64 == 0 && !kIntWide) {
        if (p.cluster_split) {
            fence_proxy_async_smem();   // the TMA-written ring now receives peers' stores
            cluster_sync_all();         // every pair's main loop is over: all rings are idle
            tc_fence_after();
            const UnitCoord c = c_first;
            if (warp >= 2 && epi_ok) {
                // rows of this CTA's half go to the CTAs (s', same half) of the cluster;
                // this warp's (idle) TMA-store buffers serve as its transpose staging
                const uint32_t stg = staging + static_cast<uint32_t>((warp - 2) * 2 * L::kStoreBufBytes);
                cluster_push_any<BN, OUT, 4>(p.split_k, ring, stg, tmem_base,
                                             ring + SplitRecv<BN>::kBytes, warp & 3, lane, c.split,
                                             2u, rank);
            }
            cluster_sync_all();         // every slice has arrived at its owner
            if (warp >= 2)
                cluster_sum_store<BN, OUT, 4>(p, c.m_blk * 2 * kBM + static_cast<int32_t>(rank) * kBM,
                                              c.n_blk * BN, static_cast<int>(crank >> 1), ring,
                                              static_cast<int>(threadIdx.x) - 64);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    cluster_sync_all();   // the pair's MMAs, TMEM reads and copies are all finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    } else if (warp >= 2) {
        // bulk stores have read their shared-memory source before the CTA ends;
        // their global writes complete with the grid
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }
}

}  // namespace gbg
