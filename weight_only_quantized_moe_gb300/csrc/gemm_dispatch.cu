// gemm_dispatch.cu - picks the GEMM instantiation and sizes its shared memory.
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i4_f16(const CUtensorMap*, const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4_bf16(const CUtensorMap*, const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8(const CUtensorMap*, const GemmParams&, int, cudaStream_t);

size_t gemm_smem_bytes(const GemmParams& p) {
  return 1024 + static_cast<size_t>(p.smem_stages) * gemm_stage_bytes(p.token_tile, p.stage_bytes) + kBarrierBytes;
}

cudaError_t launch_gemm(bool int4, bool bf16_scales, const CUtensorMap* tmap_b, const GemmParams& p, int grid,
                        cudaStream_t stream) {
  if (int4)
    return bf16_scales ? launch_gemm_i4_bf16(tmap_b, p, grid, stream) : launch_gemm_i4_f16(tmap_b, p, grid, stream);
  return launch_gemm_i8(tmap_b, p, grid, stream);
}

}  // namespace qmoe
