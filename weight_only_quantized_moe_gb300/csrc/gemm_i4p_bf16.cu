// gemm_i4p_bf16.cu - instantiation of the grouped dequant GEMM for symmetric int4 weights with bf16
// group scales applied per group in fp32 by the epilogue (16-row token tiles).
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i4p_bf16(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_gemm_t<kQ4P, true>(p, grid, stream);
}

}  // namespace qmoe
