// gemm_inst_bf16.cu -- the kernel variants with bf16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_OUTPUT(kOutBF16)
}  // namespace gbg
