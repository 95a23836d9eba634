// gemm_i8sg_bf16.cu - instantiation of the grouped dequant GEMM for 2:4-sparse int8 weights with
// bf16 group scales (one translation unit per variant so they compile in parallel).
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i8sg_bf16(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_gemm_t<kQ8SG, true>(p, grid, stream);
}

}  // namespace qmoe
