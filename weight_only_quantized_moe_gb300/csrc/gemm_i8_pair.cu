// gemm_i8_pair.cu - instantiation of the grouped dequant GEMM on CTA pairs for int8 weights with per-column scales
// (one translation unit per variant so they compile in parallel).
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i8_pair(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_gemm_t<kQ8, false, true>(p, grid, stream);
}

}  // namespace qmoe
