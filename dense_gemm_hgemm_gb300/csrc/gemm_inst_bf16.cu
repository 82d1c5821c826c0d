// gemm_inst_bf16.cu -- the one-SM kernel variants with bf16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_ONE_SM(kOutBF16)
}  // namespace gbg
