// gemm_inst_f16.cu -- instantiations and launchers of the TN GEMM kernel with
// f16 output.  Variants: (tile width BN, ring depth STAGES, k-blocks per slot; the
// depth identifies the variant).
#include "gemm_kernel.cuh"
#include "gemm_kernel_2cta.cuh"
#include "gemm_launch.h"

namespace gbg {
namespace {

template <int BN, int STAGES, int KS>
cudaError_t prepare_one(size_t* smem_bytes) {
    const size_t bytes = SmemLayout<BN, STAGES, KS>::kTotal;
    *smem_bytes = bytes;
    return cudaFuncSetAttribute(gemm_tn_kernel<BN, STAGES, kOutF16, KS>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int BN, int STAGES, int KS>
cudaError_t launch_one(const LaunchShape& s, const CUtensorMap& a, const CUtensorMap& b,
                       const CUtensorMap& c, const KParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(s.block));
    cfg.dynamicSmemBytes = s.smem_bytes;
    cfg.stream = stream;
    // Programmatic dependent launch: this kernel's set-up may overlap the tail
    // of the previous kernel in the stream (the kernel waits on it with
    // griddepcontrol.wait before touching global memory).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    unsigned n = 1;
    if (s.cluster > 1) {   // split-K slices of a tile as one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(s.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, gemm_tn_kernel<BN, STAGES, kOutF16, KS>, a, b, c, p);
}

template <int BN, int STAGES, int KS>
cudaError_t prepare_pair(size_t* smem_bytes) {
    const size_t bytes = SmemLayout2<BN, STAGES, KS>::kTotal;
    *smem_bytes = bytes;
    return cudaFuncSetAttribute(gemm_tn_pair_kernel<BN, STAGES, kOutF16, KS>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <int BN, int STAGES, int KS>
cudaError_t launch_pair(const LaunchShape& s, const CUtensorMap& a, const CUtensorMap& b,
                        const CUtensorMap& c, const KParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(s.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(s.block));
    cfg.dynamicSmemBytes = s.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;   // SM pairs (several with split-K)
    attr[1].val.clusterDim.x = static_cast<unsigned>(s.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tn_pair_kernel<BN, STAGES, kOutF16, KS>, a, b, c, p);
}

}  // namespace

cudaError_t gemm_prepare_pair_f16(int bn, int stages, size_t* smem_bytes) {
#define X(B, S, K) \
    if (bn == B && stages == S) return prepare_pair<B, S, K>(smem_bytes);
    X(256, 6, 1) X(128, 8, 1) X(256, 3, 2) X(128, 4, 2)
#undef X
    return cudaErrorInvalidValue;
}

cudaError_t gemm_launch_pair_f16(int bn, int stages, const LaunchShape& s, const CUtensorMap& a,
                              const CUtensorMap& b, const CUtensorMap& c, const KParams& p,
                              cudaStream_t stream) {
#define X(B, S, K) \
    if (bn == B && stages == S) return launch_pair<B, S, K>(s, a, b, c, p, stream);
    X(256, 6, 1) X(128, 8, 1) X(256, 3, 2) X(128, 4, 2)
#undef X
    return cudaErrorInvalidValue;
}

cudaError_t gemm_prepare_f16(int bn, int stages, size_t* smem_bytes) {
#define X(B, S, K) \
    if (bn == B && stages == S) return prepare_one<B, S, K>(smem_bytes);
    X(64, 8, 1) X(128, 6, 1) X(256, 4, 1) X(64, 4, 2) X(128, 3, 2)
#undef X
    return cudaErrorInvalidValue;
}

cudaError_t gemm_launch_f16(int bn, int stages, const LaunchShape& s, const CUtensorMap& a,
                             const CUtensorMap& b, const CUtensorMap& c, const KParams& p,
                             cudaStream_t stream) {
#define X(B, S, K) \
    if (bn == B && stages == S) return launch_one<B, S, K>(s, a, b, c, p, stream);
    X(64, 8, 1) X(128, 6, 1) X(256, 4, 1) X(64, 4, 2) X(128, 3, 2)
#undef X
    return cudaErrorInvalidValue;
}

const void* gemm_kernel_ptr_f16(int bn, int stages, int pair) {
#define X(B, S, K) \
    if (!pair && bn == B && stages == S) \
        return reinterpret_cast<const void*>(gemm_tn_kernel<B, S, kOutF16, K>);
    X(64, 8, 1) X(128, 6, 1) X(256, 4, 1) X(64, 4, 2) X(128, 3, 2)
#undef X
#define X(B, S, K) \
    if (pair && bn == B && stages == S) \
        return reinterpret_cast<const void*>(gemm_tn_pair_kernel<B, S, kOutF16, K>);
    X(256, 6, 1) X(128, 8, 1) X(256, 3, 2) X(128, 4, 2)
#undef X
    return nullptr;
}

}  // namespace gbg
