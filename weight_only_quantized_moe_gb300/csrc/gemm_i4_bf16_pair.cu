// gemm_i4_bf16_pair.cu - instantiation of the grouped dequant GEMM on CTA pairs for int4 weights with bf16 group scales
// (one translation unit per variant so they compile in parallel).
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i4_bf16_pair(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_gemm_t<kQ4, true, true>(p, grid, stream);
}

}  // namespace qmoe
