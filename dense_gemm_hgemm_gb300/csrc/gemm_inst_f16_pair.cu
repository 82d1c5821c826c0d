// gemm_inst_f16_pair.cu -- the SM-pair kernel variants with fp16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_PAIR(kOutF16)
}  // namespace gbg
