// gemm_inst_i32.cu -- the kernel variants with int32 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_OUTPUT(kOutI32)
}  // namespace gbg
