// gemm_inst.cuh -- the kernel variants (shared-memory set-up and host stub of
// each), one template per output type and kernel: gemm_inst_<type>.cu and
// gemm_inst_<type>_pair.cu instantiate the one-SM and the SM-pair half for fp16,
// bf16 and int32 output, so the six compile in parallel.  The launches
// themselves go through the plan's driver function handle.
//
// A variant is (tile width BN, ring depth STAGES, k-blocks per slot KS) of the
// one-SM kernel or of the SM-pair kernel; (BN, STAGES) identifies it, because
// every KS has its own depth for a given BN.  Each variant is compiled in the
// general form and, where a plan can use them, in the plain, cluster-split and
// epilogue forms (KernelForm).  The integer output mode keeps its int32 sums in
// registers: the one-SM kernel has the narrower variants only, and only the
// general form (the plain forms spill there); the SM-pair kernel has them all
// (224/256-wide integer tiles with eight epilogue warps).  The 224-wide SM-pair
// tile (K-contiguous B, no K split or multicast) fills the last wave of SM pairs
// on shapes whose 256-wide tile count leaves most of it idle.
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
// Forms compiled per one-SM variant: the four-k-block variant (never chosen by
// the table) and the integer mode (no fused epilogue) have the general form only.
template <int OUT, int KS, int FORM>
constexpr bool one_sm_form_ok() {
    return FORM == kFormGeneral || (OUT != kOutI32 && KS != 4);
}
// (the 128-wide integer tiles, whose register sums already spill a little in the
// general form, have that form only)
template <int OUT, int BN, int KS, int FORM>
constexpr bool pair_form_ok() {
    return FORM == kFormGeneral ||
           (FORM == kFormPlain && KS != 4 && !(OUT == kOutI32 && BN == 128)) ||
           (FORM == kFormEpilogue && KS != 4 && OUT != kOutI32);
}

template <bool PAIR, int BN, int STAGES, int OUT, int KS, int FORM>
const void* kernel_fn() {
    if constexpr (PAIR)
        return reinterpret_cast<const void*>(gemm_tn_pair_kernel<BN, STAGES, OUT, KS, FORM>);
    else
        return reinterpret_cast<const void*>(gemm_tn_kernel<BN, STAGES, OUT, KS, FORM>);
}

template <bool PAIR, int BN, int STAGES, int KS>
constexpr size_t smem_bytes() {
    if constexpr (PAIR)
        return SmemLayout2<BN, STAGES, KS>::kTotal;
    else
        return SmemLayout<BN, STAGES, KS>::kTotal;
}

template <bool PAIR, int BN, int STAGES, int OUT, int KS, int FORM>
cudaError_t prepare(size_t* smem) {
    *smem = smem_bytes<PAIR, BN, STAGES, KS>();
    return cudaFuncSetAttribute(kernel_fn<PAIR, BN, STAGES, OUT, KS, FORM>(),
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(*smem));
}

}  // namespace inst

// One kernel's variants: the host stub of (bn, stages, form) and, with `smem`
// non-null, its shared-memory size with the attribute set.  cudaErrorInvalidValue
// (stub: null) for a combination that is not compiled.
#define GBG_FORM_CASE(PAIR, B, S, K, F)                                         \
    if (form == F) {                                                            \
        if (smem) *st = inst::prepare<PAIR, B, S, OUT, K, F>(smem);             \
        return inst::kernel_fn<PAIR, B, S, OUT, K, F>();                        \
    }

template <int OUT>
const void* gemm_variant_one_sm(int bn, int stages, int form, size_t* smem, cudaError_t* st) {
#define X(B, S, K)                                                              \
    if constexpr (inst::one_sm_ok<OUT, B>())                                    \
        if (bn == B && stages == S) {                                           \
            if constexpr (inst::one_sm_form_ok<OUT, K, kFormPlain>())           \
                GBG_FORM_CASE(false, B, S, K, kFormPlain)                       \
            if constexpr (inst::one_sm_form_ok<OUT, K, kFormClusterSplit>())    \
                GBG_FORM_CASE(false, B, S, K, kFormClusterSplit)                \
            if constexpr (inst::one_sm_form_ok<OUT, K, kFormEpilogue>())        \
                GBG_FORM_CASE(false, B, S, K, kFormEpilogue)                    \
            GBG_FORM_CASE(false, B, S, K, kFormGeneral)                         \
        }
    GBG_ONE_SM_VARIANTS(X)
#undef X
    if (smem) *st = cudaErrorInvalidValue;
    return nullptr;
}

template <int OUT>
const void* gemm_variant_pair(int bn, int stages, int form, size_t* smem, cudaError_t* st) {
#define X(B, S, K)                                                              \
    if (bn == B && stages == S) {                                               \
        if constexpr (inst::pair_form_ok<OUT, B, K, kFormPlain>())              \
            GBG_FORM_CASE(true, B, S, K, kFormPlain)                            \
        if constexpr (inst::pair_form_ok<OUT, B, K, kFormEpilogue>())           \
            GBG_FORM_CASE(true, B, S, K, kFormEpilogue)                         \
        GBG_FORM_CASE(true, B, S, K, kFormGeneral)                              \
    }
    GBG_PAIR_VARIANTS(X)
#undef X
    if (smem) *st = cudaErrorInvalidValue;
    return nullptr;
}
#undef GBG_FORM_CASE

// One explicit instantiation per output type and kernel, in its own translation unit.
#define GBG_INSTANTIATE_ONE_SM(OUT) \
    template const void* gemm_variant_one_sm<OUT>(int, int, int, size_t*, cudaError_t*);
#define GBG_INSTANTIATE_PAIR(OUT) \
    template const void* gemm_variant_pair<OUT>(int, int, int, size_t*, cudaError_t*);

}  // namespace gbg
