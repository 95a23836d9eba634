// qmoe_internal.h - declarations shared by the host dispatcher and the CUDA
// translation units of libqmoe (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qmoe {

// Packed weight geometry (see the pack functions in api.cpp).
constexpr int kTileRows = 128;        // output features per GEMM work item (MMA M)
constexpr int kStageK = 128;          // K elements per pipeline stage (= one int4 group)
constexpr int kInt4StageBytes = 8448; // 128 rows x 128 K x 4 bit + 128 scales x 2 B
constexpr int kInt8StageBytes = 16384;
constexpr int kInt4ZpStageBytes = 8576;   // int4 block + 128 zero-point bytes
constexpr int kInt8GroupStageBytes = 16640;  // int8 block + 128 x 2 B scales
// 2:4-sparse int4: 128 rows x 64 kept codes (4 KB), their 2-bit positions (2 KB), 128 x 2 B scales
constexpr int kInt4SparseStageBytes = 6400;
// 2:4-sparse int8: 128 rows x 64 kept codes (8 KB), their 2-bit positions (2 KB); with group
// scales 128 x 2 B more (per-column scales live outside the blocks)
constexpr int kInt8SparseStageBytes = 10240;
constexpr int kInt8SparseGroupStageBytes = 10496;

// Weight formats of the GEMM kernel (template parameter).
// Per-group-scaled int4: each GEMM epilogue warp stages, for segments of kPgSeg
// pipeline stages, its 32 rows' group scales (2 bytes each) and the chunk's 16
// token-row corrections (fp32) in two shared-memory buffers of its own.
constexpr int kPgSeg = 16;
constexpr int kPgWarpBuf = kPgSeg * (32 * 2 + 16 * 4);  // one buffer: scales, then corrections
constexpr int kPgStageBytes = 4 * 2 * kPgWarpBuf;       // 4 warps x 2 buffers
// kQ4P: symmetric int4 with per-group fp32 scaling in the epilogue (kernel variant
// of kQ4 chosen by GemmParams::pg; not a storage format)
enum QuantKind : int { kQ4 = 0, kQ4Z = 1, kQ8 = 2, kQ8G = 3, kQ4S = 4, kQ8S = 5, kQ8SG = 6, kQ4P = 7 };
constexpr int kAlignBlock = 16;       // moe_align block used by the forward (the MMA N granule)
constexpr int kNoPadPairs = 8;       // batches up to this many pairs leave padding rows unwritten
constexpr int kMaxTokenTile = 256;

// Device-side status codes (values match qmoe_status).
constexpr int kStatusTimeout = 6;
constexpr int kStatusBadExpert = 7;

// One work-item row range of one expert, produced by the align kernel.
struct Chunk {
  int32_t expert;
  int32_t row0;
  int32_t nrows;  // multiple of 16, <= token tile
  int32_t first;  // index of the expert's first chunk
  int32_t count;  // chunks of the expert
  int32_t pad;
};

enum EpiMode : int32_t {
  kEpiSiluToAct = 0,   // gate/up GEMM, whole K: fp32 inter[row, j] = SiLU(gate)*up
  kEpiPartialRows = 1, // gate/up GEMM or dense linear, split K: fp32 partial [split][row][N]
  kEpiWeightedPairs = 2, // down GEMM: fp32 y[split][pair][H] = topk_weight * acc
  kEpiLinearOut = 3    // dense linear, whole K: out[row, n] in the activation type, rows < P
};

// Pre-staged B operand (the gathered activations, the f16 intermediate): K is
// cut into 128-K groups; group u holds all cap rows (cap a multiple of 16) as
// [row / 8][64-K block][row % 8][128 B], the eight 16-byte pieces of every
// 128-byte row XOR-swizzled by row % 8 (the 128-byte swizzle of a K-major MMA
// operand).  A chunk's rows of one group are one contiguous run of
// nrows * 256 bytes.  Byte offset of the piece holding elements k..k+7
// (k % 8 == 0) of row r:
__host__ __device__ inline int64_t staged_offset(int64_t r, int k, int64_t cap) {
  const int unit = k >> 7, blk = (k >> 6) & 1, piece = (k & 63) >> 3;
  const int sw = static_cast<int>(r & 7);
  return static_cast<int64_t>(unit) * cap * 256 + (r >> 3) * 2048 + blk * 1024 + sw * 128 + ((piece ^ sw) << 4);
}

struct GemmParams {
  const uint8_t* w;          // packed weights [E][n_tiles][k_groups][stage_bytes]
  const uint8_t* b;          // pre-staged B operand (see staged_offset)
  const float* row_scale;    // int8: per packed row [E][n_tiles*128]; int4: null
  const float* col_scale;    // per B row (token row): 2^e of its power-of-two f16 scaling
  const Chunk* chunks;       // [max_chunks]
  const int32_t* n_chunks;   // device scalar
  const int32_t* sorted_ids; // down GEMM epilogue
  const float* topk_w;       // flat [P]
  void* out;
  int32_t* status;
  int64_t out_ld;            // elements per output row
  int64_t out_split_stride;  // elements per split slab
  int64_t b_unit_stride;     // bytes per 128-K group of the staged B operand (cap * 256)
  int32_t n_tiles;
  int32_t k_groups;          // 128-K quantization groups along K = pipeline stages per tile
  int32_t split;
  int32_t token_tile;        // T: B rows per stage buffer, TMEM columns per accumulator
  int32_t acc_bufs;          // TMEM accumulators per MMA issuer (1 or 2)
  int32_t issuers;           // MMA-issuing warps (1 to 3)
  int32_t a_col0;            // first TMEM column of the A slots
  int32_t w_stages;          // packed-weight ring depth (even)
  int32_t ab_stages;         // TMEM A slots of 64 columns (even)
  int32_t b_stages;          // token-tile ring depth in shared memory (a multiple of ab_stages)
  int32_t stage_bytes;       // packed weight bytes per 128-K group
  int32_t epi_mode;
  int32_t P;                 // number of token-expert pairs
  int32_t chunk_group;       // work-item raster: chunks per group (> 0), or -G: pieces of at most G chunks of one expert
  int32_t inter_ld;          // I (for the SiLU epilogue)
  int32_t fault_injection;   // 1: CTA 0 arms its first stage without copies (failure-path test)
  int32_t out_bf16;          // kEpiLinearOut: output type bf16 (else f16)
  int32_t dq_sets;           // dequant sets (2 of 8 half-row warps, or 4 of 4 full-row warps)
  int32_t w_shared;          // 1: an expert's weight tiles are read by several chunks (L2 evict-normal)
  int32_t pg;                // int4, 16-row tiles: raw magic-number A, per-stage D slots, per-group fp32 scaling
  int32_t pair;              // clusters of two CTAs: M = 256 MMAs over both SMs, each CTA with half the token rows
  int32_t d_col0;            // per-group scaling: first TMEM column of the 16-column D slots (one per A slot)
  const float* pg_corr;      // per-group scaling: token-row corrections [k_groups][pg_cap]
  int64_t pg_cap;
  // down GEMM with the top-k reduction in its epilogue (red_cnt null: a separate
  // kernel sums the partial outputs)
  int32_t* red_cnt;          // [M][n_tiles][4] arrival counters, zero at launch
  const int32_t* topk_ids;   // [M][top_k]
  uint16_t* red_out;         // [M][out_ld] layer output in the activation type (out_bf16)
  int32_t top_k;
  int32_t n_experts;
};

// Launch with programmatic stream serialization when `pdl` is set: the kernel
// may start while the previous kernel in the stream finishes; it must execute
// griddepcontrol.wait before reading that kernel's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of `cluster_x` CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t stream, bool pdl, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Host-side launchers (defined in the .cu files); return cudaError_t of the launch.
cudaError_t launch_align(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block, int64_t capacity,
                         int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded, int32_t token_tile,
                         Chunk* chunks, int32_t* n_chunks, int32_t* status, cudaStream_t stream);

cudaError_t launch_gather(const void* x, bool bf16, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* num_post_padded, const int32_t* perm13, int32_t P, int32_t top_k,
                          int32_t H, int32_t block, int64_t cap_rows, void* xg, float* xscale, float* pg_corr,
                          int num_sms, cudaStream_t stream);

// moe_align and the gather fused for small batches (P <= 1024 pairs, shared memory permitting).
bool align_gather_small_fits(int32_t P, int32_t E, int32_t block, int32_t H, bool act_order);
cudaError_t launch_align_gather_small(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block, int64_t capacity,
                                      int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                      int32_t token_tile, Chunk* chunks, int32_t* n_chunks, int32_t* status,
                                      const void* x, bool bf16, const int32_t* perm13, int32_t top_k, int32_t H,
                                      int64_t cap_rows, void* xg, float* xscale, float* pg_corr, int num_sms,
                                      cudaStream_t stream);

cudaError_t launch_silu_reduce(const float* h, const int32_t* num_post_padded, int32_t split, int64_t cap_rows,
                               int32_t I, float* inter32, int num_sms, cudaStream_t stream);

// Preparation of the down GEMM's in-epilogue top-k reduction, done by the
// intermediate rescale kernel (null cnt: none): zero the arrival counters, and
// write zero output rows for tokens with no valid expert (no GEMM item reaches them).
struct TopkPrep {
  int32_t* cnt;
  int64_t n_cnt;
  const int32_t* topk_ids;
  int64_t M;
  int32_t top_k;
  int32_t E;
  int32_t H;
  uint16_t* out;
};
cudaError_t launch_inter_rescale(const float* inter32, const int32_t* num_post_padded, const int32_t* sorted_ids,
                                 int32_t P, int32_t I, int64_t cap_rows, void* inter16, float* iscale, float* pg_corr,
                                 const TopkPrep& prep, int num_sms, cudaStream_t stream);

cudaError_t launch_out_reduce(const float* y, const int32_t* topk_ids, int32_t E, int32_t split, int64_t M,
                              int32_t top_k, int32_t H, bool bf16, void* out, int num_sms, cudaStream_t stream);

// Dense linear, split K: out[m, n] = sum_s h[s, m, n] (fp32 partials, slabs of cap_rows x N) cast to the
// activation type, m < M.
cudaError_t launch_linear_reduce(const float* h, int32_t split, int64_t cap_rows, int64_t M, int32_t N, bool bf16,
                                 void* out, int num_sms, cudaStream_t stream);

// dtype: 0 f32, 1 f16, 2 bf16 logits; 1 <= E <= 1024, 1 <= k <= min(E, 32).
cudaError_t launch_route_topk(const void* logits, int dtype, int64_t M, int32_t E, int32_t k, int32_t renormalize,
                              int32_t* topk_ids, float* topk_weights, int num_sms, cudaStream_t stream);

size_t gemm_smem_bytes(const GemmParams& p);
cudaError_t launch_gemm(QuantKind kind, bool bf16_scales, const GemmParams& p, int grid, cudaStream_t stream);

}  // namespace qmoe

#include "qmoe.h"

namespace qmoe {
// The forward on a caller-supplied device workspace of ws_bytes bytes (api.cpp).
qmoe_status forward_into_workspace(const qmoe_layer* layer, const void* x, int64_t M, const int32_t* topk_ids,
                                   const float* topk_weights, int32_t top_k, void* out, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);
}  // namespace qmoe
