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
constexpr int default_pair_stages_ks2(int bn) { return bn >= 224 ? 3 : 4; }
constexpr int default_pair_stages(int bn) { return bn >= 224 ? 6 : 8; }
// Four k-blocks per ring slot (one-SM BN 64, SM-pair BN 128): two 96 KiB slots.
constexpr int default_stages_ks4(int) { return 2; }
// Ring depth of a variant: one-SM or pair kernel, tile width, k-blocks per slot.
constexpr int default_ring_stages(int pair, int bn, int ks) {
    return ks == 4 ? default_stages_ks4(bn)
           : pair  ? (ks == 2 ? default_pair_stages_ks2(bn) : default_pair_stages(bn))
                   : (ks == 2 ? default_stages_ks2(bn) : default_stages(bn));
}

struct LaunchShape {
    int grid;
    int block;
    size_t smem_bytes;
    int cluster = 1;   // CTAs per thread-block cluster (x dimension)
};

// Kernel variant lookup.  `out` is kOutF16 / kOutBF16 / kOutI32, `pair` = 1 for
// the SM-pair kernel, `form` a KernelForm.  gemm_prepare: cudaErrorInvalidValue
// if the variant (bn, stages, out, pair, form) is not compiled, else its
// shared-memory size (and the attribute set); gemm_kernel_ptr: the variant's
// host stub, or null.  A launch passes the kernel the three tensor maps and the
// KParams block, in that order.
cudaError_t gemm_prepare(int bn, int stages, int out, int pair, int form, size_t* smem_bytes);
const void* gemm_kernel_ptr(int bn, int stages, int out, int pair, int form);

// Per output type and kernel (defined in gemm_inst.cuh, instantiated in
// gemm_inst_<type>.cu and gemm_inst_<type>_pair.cu): the host stub, and with
// `smem` non-null the shared-memory size and the attribute's status in *st.
template <int OUT>
const void* gemm_variant_one_sm(int bn, int stages, int form, size_t* smem, cudaError_t* st);
template <int OUT>
const void* gemm_variant_pair(int bn, int stages, int form, size_t* smem, cudaError_t* st);

// Co-resident clusters of shape.cluster CTAs of a kernel variant.
cudaError_t gemm_max_clusters(int bn, int stages, int out, int pair, int form,
                              const LaunchShape& shape, int* n);

// Auxiliary kernels (gemm_aux.cu).
cudaError_t launch_widen_i8(const int8_t* a, int64_t na, const int8_t* b, int64_t nb, void* a16,
                            void* b16, int num_sms, cudaStream_t stream);
cudaError_t launch_zero_fill(void* dst, int64_t bytes, int num_sms, cudaStream_t stream);
cudaError_t launch_empty(int grid, cudaStream_t stream);
cudaError_t launch_fill_bias_act(void* C, int64_t M, int64_t N, const float* bias, int act,
                                 int bf16, int num_sms, cudaStream_t stream);

}  // namespace gbg
