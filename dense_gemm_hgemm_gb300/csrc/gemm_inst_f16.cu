// gemm_inst_f16.cu -- the kernel variants with fp16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_OUTPUT(kOutF16)
}  // namespace gbg
