// gemm_inst_bf16_pair.cu -- the SM-pair kernel variants with bf16 output (see gemm_inst.cuh).
#include "gemm_inst.cuh"

namespace gbg {
GBG_INSTANTIATE_PAIR(kOutBF16)
}  // namespace gbg
