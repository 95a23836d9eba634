// gemm_dispatch.cu - picks the GEMM instantiation and sizes its shared memory.
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i4_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8(const GemmParams&, int, cudaStream_t);

size_t gemm_smem_bytes(const GemmParams& p) {
  return 1024 + static_cast<size_t>(p.smem_stages) * gemm_stage_bytes(p.token_tile, p.stage_bytes, p.ks) + kBarrierBytes;
}

cudaError_t launch_gemm(bool int4, bool bf16_scales, const GemmParams& p, int grid,
                        cudaStream_t stream) {
  // the even/odd role split needs rings of even size (see qmoe_gemm_kernel)
  if (p.smem_stages < 2 || p.a_stages < 2 || (p.smem_stages & 1) || (p.a_stages & 1)) return cudaErrorInvalidValue;
  if (int4)
    return bf16_scales ? launch_gemm_i4_bf16(p, grid, stream) : launch_gemm_i4_f16(p, grid, stream);
  return launch_gemm_i8(p, grid, stream);
}

}  // namespace qmoe
