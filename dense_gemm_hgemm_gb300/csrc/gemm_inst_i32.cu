// gemm_inst_i32.cu -- the one-SM kernel variants with int32 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_ONE_SM(kOutI32)
}  // namespace gbg
