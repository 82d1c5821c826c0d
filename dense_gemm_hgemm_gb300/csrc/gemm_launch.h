// gemm_launch.h -- host-side entry points of the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_kernel_params.h"

namespace gbg {

// Default ring depth per tile width (all near 192 KiB of the 227 KiB a CTA may use).
constexpr int default_stages(int bn) { return bn == 256 ? 4 : (bn == 128 ? 6 : 8); }
// Two k-blocks per ring slot (one-SM kernel, BN 64 / 128): the same ~192 KiB ring.
constexpr int default_stages_ks2(int bn) { return bn == 128 ? 3 : 4; }
// SM-pair kernel: each CTA holds A 128 x 64 and half of B per stage.
constexpr int default_pair_stages_ks2(int bn) { return bn == 256 ? 3 : 4; }
constexpr int default_pair_stages(int bn) { return bn == 256 ? 6 : 8; }

struct LaunchShape {
    int grid;
    int block;
    size_t smem_bytes;
    int cluster = 1;   // CTAs per thread-block cluster (x dimension)
};

// Kernel variant lookup.  `out` is kOutF16 / kOutBF16 / kOutI32.  Returns
// cudaErrorInvalidValue if no variant exists for (bn, stages, out).
cudaError_t gemm_prepare(int bn, int stages, int out, size_t* smem_bytes);
cudaError_t gemm_launch(int bn, int stages, int out, const LaunchShape& shape,
                        const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                        const CUtensorMap& tmap_c, const KParams& p, cudaStream_t stream);

// Per-output-type translation units.
cudaError_t gemm_prepare_f16(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_prepare_bf16(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_prepare_i32(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_launch_f16(int bn, int stages, const LaunchShape&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const KParams&, cudaStream_t);
cudaError_t gemm_launch_bf16(int bn, int stages, const LaunchShape&, const CUtensorMap&, const CUtensorMap&,
                             const CUtensorMap&, const KParams&, cudaStream_t);
cudaError_t gemm_launch_i32(int bn, int stages, const LaunchShape&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const KParams&, cudaStream_t);

// Co-resident clusters of shape.cluster CTAs of a kernel variant (pair = 1: the
// SM-pair kernel).
cudaError_t gemm_max_clusters(int bn, int stages, int out, int pair, const LaunchShape& shape,
                              int* n);
const void* gemm_kernel_ptr_f16(int bn, int stages, int pair);
const void* gemm_kernel_ptr_bf16(int bn, int stages, int pair);
const void* gemm_kernel_ptr_i32(int bn, int stages, int pair);

// SM-pair (cta_group::2) kernels, 16-bit outputs.
cudaError_t gemm_prepare_pair_f16(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_prepare_pair_bf16(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_launch_pair_f16(int bn, int stages, const LaunchShape&, const CUtensorMap&,
                                 const CUtensorMap&, const CUtensorMap&, const KParams&, cudaStream_t);
cudaError_t gemm_prepare_pair_i32(int bn, int stages, size_t* smem_bytes);
cudaError_t gemm_launch_pair_i32(int bn, int stages, const LaunchShape&, const CUtensorMap&,
                                 const CUtensorMap&, const CUtensorMap&, const KParams&, cudaStream_t);
cudaError_t gemm_launch_pair_bf16(int bn, int stages, const LaunchShape&, const CUtensorMap&,
                                  const CUtensorMap&, const CUtensorMap&, const KParams&,
                                  cudaStream_t);

// Auxiliary kernels (gemm_aux.cu).
cudaError_t launch_widen_i8(const int8_t* a, int64_t na, const int8_t* b, int64_t nb, void* a16,
                            void* b16, int num_sms, cudaStream_t stream);
cudaError_t launch_zero_fill(void* dst, int64_t bytes, int num_sms, cudaStream_t stream);
cudaError_t launch_empty(int grid, cudaStream_t stream);
cudaError_t launch_fill_bias_act(void* C, int64_t M, int64_t N, const float* bias, int act,
                                 int bf16, int num_sms, cudaStream_t stream);

}  // namespace gbg
