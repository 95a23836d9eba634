// gemm_dispatch.cu - picks the GEMM instantiation and sizes its shared memory.
#include "gemm.cuh"

namespace qmoe {

cudaError_t launch_gemm_i4_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4p_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4p_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4z_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4z_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4s_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4s_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8g_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8g_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8s(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8sg_f16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8sg_bf16(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4_f16_pair(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i4_bf16_pair(const GemmParams&, int, cudaStream_t);
cudaError_t launch_gemm_i8_pair(const GemmParams&, int, cudaStream_t);

size_t gemm_smem_bytes(const GemmParams& p) {
  return gemm_smem_layout_bytes(p.w_stages, p.stage_bytes, p.b_stages, p.token_tile, p.pg != 0, p.pair != 0);
}

cudaError_t launch_gemm(QuantKind kind, bool bf16_scales, const GemmParams& p, int grid, cudaStream_t stream) {
  // ring sizes must be multiples of every role's stride (see qmoe_gemm_kernel)
  if (p.issuers < 1 || p.issuers > kMaxIssuers) return cudaErrorInvalidValue;
  const int mult = (p.issuers == 3) ? 6 : 2;
  if (p.w_stages < 2 || (p.w_stages & 1) || p.ab_stages < mult || p.ab_stages % mult != 0) return cudaErrorInvalidValue;
  if (p.b_stages < p.ab_stages || p.b_stages % p.ab_stages != 0) return cudaErrorInvalidValue;
  // dequant sets: each weight slot and each token-tile ("done") barrier must belong to one set
  if (p.dq_sets != 2 && p.dq_sets != 4) return cudaErrorInvalidValue;
  // every role starts at ring position = its index and steps by its stride with
  // one wrap: each ring holds at least as many slots as the stride of its users
  if (p.ab_stages < p.dq_sets || p.ab_stages < p.issuers || p.w_stages < p.dq_sets) return cudaErrorInvalidValue;
  // per-group scaling: 16-row tiles, at most 8 A slots, D slots after the A slots within 512 columns
  if (p.pg && (kind != kQ4 || p.token_tile != 16 || p.ab_stages > 8 || p.pg_corr == nullptr ||
               p.d_col0 < p.a_col0 + 64 * p.ab_stages || p.d_col0 + 16 * p.ab_stages > 512))
    return cudaErrorInvalidValue;
  if (p.w_stages % p.dq_sets != 0 || p.b_stages % p.dq_sets != 0) return cudaErrorInvalidValue;
  // barriers (2 per weight slot, 1 per A slot, 1 per token-tile slot, 4 + kMaxIssuers more),
  // the TMEM address and the abort flag fit the barrier area
  if ((2 * p.w_stages + p.ab_stages + p.b_stages + 4 + kMaxIssuers) * 8 + 8 > kBarrierBytes)
    return cudaErrorInvalidValue;
  // CTA pairs: dense int4 (symmetric) and per-column int8 with the standard epilogue and
  // the separate top-k reduction; token tiles whose halves are whole 8-row groups
  if (p.pair) {
    if (p.pg || p.red_cnt != nullptr || p.token_tile % 16 != 0) return cudaErrorInvalidValue;
    if (kind == kQ4) return bf16_scales ? launch_gemm_i4_bf16_pair(p, grid, stream) : launch_gemm_i4_f16_pair(p, grid, stream);
    if (kind == kQ8) return launch_gemm_i8_pair(p, grid, stream);
    return cudaErrorInvalidValue;
  }
  switch (kind) {
    case kQ4:
      if (p.pg) return bf16_scales ? launch_gemm_i4p_bf16(p, grid, stream) : launch_gemm_i4p_f16(p, grid, stream);
      return bf16_scales ? launch_gemm_i4_bf16(p, grid, stream) : launch_gemm_i4_f16(p, grid, stream);
    case kQ4Z: return bf16_scales ? launch_gemm_i4z_bf16(p, grid, stream) : launch_gemm_i4z_f16(p, grid, stream);
    case kQ8G: return bf16_scales ? launch_gemm_i8g_bf16(p, grid, stream) : launch_gemm_i8g_f16(p, grid, stream);
    case kQ4S: return bf16_scales ? launch_gemm_i4s_bf16(p, grid, stream) : launch_gemm_i4s_f16(p, grid, stream);
    case kQ8S: return launch_gemm_i8s(p, grid, stream);
    case kQ8SG: return bf16_scales ? launch_gemm_i8sg_bf16(p, grid, stream) : launch_gemm_i8sg_f16(p, grid, stream);
    default: return launch_gemm_i8(p, grid, stream);
  }
}

}  // namespace qmoe
