// gemm_inst_f16.cu -- the one-SM kernel variants with fp16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_ONE_SM(kOutF16)
}  // namespace gbg
