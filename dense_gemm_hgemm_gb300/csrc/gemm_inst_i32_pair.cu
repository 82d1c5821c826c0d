// gemm_inst_i32_pair.cu -- the SM-pair kernel variants with int32 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_PAIR(kOutI32)
}  // namespace gbg
