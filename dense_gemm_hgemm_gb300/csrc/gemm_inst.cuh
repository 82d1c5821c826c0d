// gemm_inst.cuh -- the kernel variants (shared-memory set-up and host stub of
// each), one template per output type (gemm_inst_f16.cu, gemm_inst_bf16.cu and
// gemm_inst_i32.cu each instantiate it once, so the three compile in parallel).
// The launches themselves go through the plan's driver function handle.
//
// A variant is (tile width BN, ring depth STAGES, k-blocks per slot KS) of the
// one-SM kernel or of the SM-pair kernel; (BN, STAGES) identifies it, because
// every KS has its own depth for a given BN.  The integer output mode keeps its int32 sums
// in registers: the one-SM kernel has the narrower variants only, the SM-pair kernel all of
// them (224/256-wide integer tiles with eight epilogue warps).  The 224-wide SM-pair tile
// (K-contiguous B, no K split or multicast) fills the last wave of SM pairs on shapes whose
// 256-wide tile count leaves most of it idle.
#pragma once

#include "gemm_kernel.cuh"
#include "gemm_kernel_2cta.cuh"
#include "gemm_launch.h"

// X(BN, STAGES, KS) for every variant of each kernel.
#define GBG_ONE_SM_VARIANTS(X) \
    X(64, 8, 1) X(128, 6, 1) X(256, 4, 1) X(64, 4, 2) X(128, 3, 2) X(64, 2, 4)
#define GBG_PAIR_VARIANTS(X) \
    X(256, 6, 1) X(224, 6, 1) X(128, 8, 1) X(256, 3, 2) X(224, 3, 2) X(128, 4, 2) X(128, 2, 4)

namespace gbg {
namespace inst {

template <int OUT, int BN>
constexpr bool one_sm_ok() { return OUT != kOutI32 || BN <= 128; }
template <int OUT, int BN>
constexpr bool pair_ok() { return true; }

template <bool PAIR, int BN, int STAGES, int OUT, int KS, bool PLAIN>
const void* kernel_fn() {
    if constexpr (PAIR)
        return reinterpret_cast<const void*>(gemm_tn_pair_kernel<BN, STAGES, OUT, KS>);
    else
        return reinterpret_cast<const void*>(gemm_tn_kernel<BN, STAGES, OUT, KS, PLAIN>);
}

template <bool PAIR, int BN, int STAGES, int KS>
constexpr size_t smem_bytes() {
    if constexpr (PAIR)
        return SmemLayout2<BN, STAGES, KS>::kTotal;
    else
        return SmemLayout<BN, STAGES, KS>::kTotal;
}

template <bool PAIR, int BN, int STAGES, int OUT, int KS, bool PLAIN>
cudaError_t prepare(size_t* smem) {
    *smem = smem_bytes<PAIR, BN, STAGES, KS>();
    return cudaFuncSetAttribute(kernel_fn<PAIR, BN, STAGES, OUT, KS, PLAIN>(),
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(*smem));
}

}  // namespace inst

// `plain` selects the one-SM kernel's plain form (gemm_tn_kernel<..., true>,
// fp16/bf16 output; the integer mode's register sums leave it no room); the
// SM-pair kernel has one form.
template <int OUT>
cudaError_t gemm_prepare_out(int bn, int stages, int pair, int plain, size_t* smem) {
#define X(B, S, K)                                                              \
    if constexpr (inst::one_sm_ok<OUT, B>())                                    \
        if (!pair && bn == B && stages == S) {                                  \
            if constexpr (OUT != kOutI32)                                       \
                if (plain) return inst::prepare<false, B, S, OUT, K, true>(smem); \
            return inst::prepare<false, B, S, OUT, K, false>(smem);             \
        }
    GBG_ONE_SM_VARIANTS(X)
#undef X
#define X(B, S, K)                                                              \
    if constexpr (inst::pair_ok<OUT, B>())                                      \
        if (pair && bn == B && stages == S) return inst::prepare<true, B, S, OUT, K, false>(smem);
    GBG_PAIR_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

template <int OUT>
const void* gemm_kernel_ptr_out(int bn, int stages, int pair, int plain) {
#define X(B, S, K)                                                              \
    if constexpr (inst::one_sm_ok<OUT, B>())                                    \
        if (!pair && bn == B && stages == S) {                                  \
            if constexpr (OUT != kOutI32)                                       \
                if (plain) return inst::kernel_fn<false, B, S, OUT, K, true>(); \
            return inst::kernel_fn<false, B, S, OUT, K, false>();               \
        }
    GBG_ONE_SM_VARIANTS(X)
#undef X
#define X(B, S, K)                                                              \
    if constexpr (inst::pair_ok<OUT, B>())                                      \
        if (pair && bn == B && stages == S) return inst::kernel_fn<true, B, S, OUT, K, false>();
    GBG_PAIR_VARIANTS(X)
#undef X
    return nullptr;
}

// One explicit instantiation per output type, in that type's translation unit.
#define GBG_INSTANTIATE_OUTPUT(OUT)                                                        \
    template cudaError_t gemm_prepare_out<OUT>(int, int, int, int, size_t*);              \
    template const void* gemm_kernel_ptr_out<OUT>(int, int, int, int);

}  // namespace gbg
