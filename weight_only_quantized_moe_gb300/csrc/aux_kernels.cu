// aux_kernels.cu - the non-GEMM steps of the fused MoE layer on sm_103a:
//   moe_align_block_size  (group token-expert pairs by expert, pad to the block)
//   token gather          (sorted, padded, act-order-permuted activation rows)
//   split-K SiLU reduce   (sum gate/up partials, apply SiLU(gate)*up)
//   intermediate rescale  (fp32 intermediate -> per-row scaled f16 for the down GEMM)
//   output reduce         (sum the top-k weighted expert outputs per token)
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qmoe_internal.h"

namespace qmoe {

// ---------------------------------------------------------------------------
// moe_align_block_size
//
// Page "Marlin moe integration" (review thread): the fused kernel relies on
// moe_align_block_size_kernel, which groups the token-expert pairs of each
// expert and pads every group to the kernel's block size (16 there).  This
// version is one CTA of 32 warps and is deterministic and stable: each warp
// owns a contiguous segment of pairs; warp-level __match_any_sync groups the
// lanes of one iteration by expert, so a warp counts and later places its
// pairs without atomics, in pair order; per-(warp, expert) write cursors come
// from a scan over experts and warps.
// ---------------------------------------------------------------------------
constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

// Exclusive block-wide scan of one value per thread (1024 threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[31];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kAlignThreads, 1)
    moe_align_kernel(const int32_t* __restrict__ ids, int32_t P, int32_t E, int32_t B, int64_t capacity,
                     int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                     int32_t* __restrict__ num_post_padded, int32_t T, Chunk* __restrict__ chunks,
                     int32_t* __restrict__ n_chunks, int32_t* __restrict__ status) {
  extern __shared__ int32_t sm[];
  int32_t* cur = sm;                     // [warps][E]: counts, then write cursors
  __shared__ int warp_sums[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel in the stream has completed (no-op without PDL)

  if (tid == 0) {
    s_bad = 0;
    if (status != nullptr) *status = 0;  // first kernel of a forward: clear its fault word
  }
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cur[i] = 0;
  __syncthreads();

  // 1. per-warp, per-expert counts over a contiguous segment of pairs
  const int seg = (P + kAlignWarps - 1) / kAlignWarps;
  const int beg = warp * seg;
  const int end = min(P, beg + seg);
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    const bool in = p < end;
    const int e = in ? (ids != nullptr ? __ldg(ids + p) : 0) : -1;  // no ids: every pair is expert 0
    const bool valid = in && e >= 0 && e < E;
    if (in && !valid) s_bad = 1;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(peers) - 1) cur[warp * E + e] += __popc(peers);
  }
  __syncthreads();

  // 2. totals, padded sizes and offsets per expert (one thread per expert)
  const int e = tid;
  int tot = 0;
  if (e < E) {
    for (int w = 0; w < kAlignWarps; ++w) tot += cur[w * E + e];
  }
  const int pad = (tot + B - 1) / B * B;
  int total;
  const int off = block_exclusive_scan(e < E ? pad : 0, warp_sums, &total);
  const int nch = (e < E && T > 0) ? (pad + T - 1) / T : 0;
  int total_chunks;
  const int coff = block_exclusive_scan(nch, warp_sums, &total_chunks);
  if (e < E) {
    int run = off;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = cur[w * E + e];
      cur[w * E + e] = run;
      run += c;
    }
    // padding slots of this expert, its block -> expert entries, its chunks
    for (int i = off + tot; i < off + pad; ++i) sorted_ids[i] = P;
    for (int b = off / B; b < (off + pad) / B; ++b) expert_ids[b] = e;
    for (int c = 0; c < nch; ++c) {
      Chunk ch;
      ch.expert = e;
      ch.row0 = off + c * T;
      ch.nrows = min(T, pad - c * T);
      ch.first = coff;
      ch.count = nch;
      ch.pad = 0;
      chunks[coff + c] = ch;
    }
  }
  // tail past the padded total
  for (int64_t i = total + tid; i < capacity; i += kAlignThreads) sorted_ids[i] = P;
  const int64_t nblocks = (capacity + B - 1) / B;
  for (int64_t b = total / B + tid; b < nblocks; b += kAlignThreads) expert_ids[b] = -1;
  __syncthreads();

  // 3. stable scatter: each warp re-walks its segment in pair order
  for (int base = beg; base < end; base += 32) {
    const int p = base + lane;
    const bool in = p < end;
    const int ex = in ? (ids != nullptr ? __ldg(ids + p) : 0) : -1;
    const bool valid = in && ex >= 0 && ex < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? ex : -1);
    if (valid) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      sorted_ids[cur[warp * E + ex] + rank] = p;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) cur[warp * E + ex] += __popc(peers);
    __syncwarp();
  }

  if (tid == 0) {
    *num_post_padded = total;
    if (n_chunks != nullptr) *n_chunks = total_chunks;
    if (s_bad && status != nullptr) atomicCAS(status, 0, kStatusBadExpert);
  }
}

cudaError_t launch_align(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block, int64_t capacity,
                         int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded, int32_t token_tile,
                         Chunk* chunks, int32_t* n_chunks, int32_t* status, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kAlignWarps) * E * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(moe_align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  // first kernel of a forward (batches above the fused kernel's size): plain
  // stream order behind the caller's work
  return launch_kernel(moe_align_kernel, dim3(1), dim3(kAlignThreads), smem, stream, false, topk_ids, P, E, block,
                       capacity, sorted_ids, expert_ids, num_post_padded, chunks ? token_tile : 0, chunks, n_chunks,
                       status);
}

// ---------------------------------------------------------------------------
// Per-row power-of-two scaling into f16.
//
// Both GEMMs multiply in f16 (11-bit significand) whatever the activation type:
// a bf16 row (8-bit significand) times a power of two is exact in f16 as long as
// it stays in f16's normal range, so each row r is stored as v * 2^-e_r with
// e_r = floor(log2 max|v|) - 14 (the row's largest magnitude lands in
// [2^14, 2^15)) and 2^e_r is kept beside it; the GEMM epilogue multiplies the
// fp32 accumulator column back by 2^e_r.  Elements below 2^-28 of the row's
// largest lose significand bits, which does not move a dot product.
// ---------------------------------------------------------------------------
// Returns (2^e, 2^-e) for a row whose largest magnitude is amax.
__device__ __forceinline__ float2 row_exponent_scale(float amax) {
  if (!(amax > 0.0f) || !(amax <= 3.4028235e38f)) return make_float2(1.0f, 1.0f);  // zero, inf or NaN
  // e in [-126, 126] keeps both 2^e and 2^-e normal fp32 numbers; then every
  // row with a normal largest magnitude above 2^-112 lands in [2^14, 2^15)
  int e = ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 14;
  e = max(-126, min(126, e));
  // both powers of two built from their exponent fields
  return make_float2(__int_as_float((127 + e) << 23), __int_as_float((127 - e) << 23));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

template <bool BF16>
__device__ __forceinline__ float act_to_float(uint16_t b) {
  if (BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  return __half2float(*reinterpret_cast<const __half*>(&b));
}

__device__ __forceinline__ uint16_t f16_bits(float v) {
  return __half_as_ushort(__float2half_rn(v));
}

// ---------------------------------------------------------------------------
// Token gather: row `row` of the gate/up GEMM's B operand is
// x[sorted_ids[row] / top_k, perm13_e] * 2^-e_row in f16, stored in the
// pre-staged layout (staged_offset), with xscale[row] = 2^e_row; padding rows
// are zeros with scale 1.  With act-order the hidden channels are put in each
// expert's sorted-group order so the GEMM walks K in whole quantization groups.
// One warp per row; lane work unit = 8 consecutive K (one 16-byte piece).
// ---------------------------------------------------------------------------
constexpr int kGatherThreads = 256;

template <bool BF16>
__device__ __forceinline__ uint4 scale_to_f16x8(const uint16_t (&e)[8], float inv) {
  uint4 o;
  o.x = static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[0]) * inv)) |
        (static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[1]) * inv)) << 16);
  o.y = static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[2]) * inv)) |
        (static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[3]) * inv)) << 16);
  o.z = static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[4]) * inv)) |
        (static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[5]) * inv)) << 16);
  o.w = static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[6]) * inv)) |
        (static_cast<uint32_t>(f16_bits(act_to_float<BF16>(e[7]) * inv)) << 16);
  return o;
}

// Token operand of the per-group-scaled int4 GEMM (16-row token tiles, symmetric
// int4): the GEMM feeds the MMA the raw magic-number halves of the codes, 1024 + q
// at input channels k with k % 4 in {0, 1} and 1024 + 16 q at k % 4 in {2, 3}, so
// the token values at the second kind are stored divided by 16 (exact, a power
// of two) and, per row and 128-channel group g, the correction
//     C[g][row] = 1032 * X_lo + 72 * X_hi,
// X_lo / X_hi = the sums of the row's stored values over the group's channels of
// each kind (the X_hi values taken before the division), satisfies
//     sum_k (q_k - 8) x_k = D - C,   D = the MMA's sum of (magic half) * (stored value).
// A 16-byte piece holds channels 8c .. 8c+7: words 1 and 3 are the divided kind.
__device__ __forceinline__ void pg_piece(uint4& o, float& xlo, float& xhi) {
  const __half2 sixteenth = __float2half2_rn(0.0625f);
  __half2 w1 = *reinterpret_cast<__half2*>(&o.y), w3 = *reinterpret_cast<__half2*>(&o.w);
  w1 = __hmul2(w1, sixteenth);
  w3 = __hmul2(w3, sixteenth);
  o.y = *reinterpret_cast<uint32_t*>(&w1);
  o.w = *reinterpret_cast<uint32_t*>(&w3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&o.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&o.z));
  const float2 c1 = __half22float2(w1), c3 = __half22float2(w3);
  xlo += (a.x + a.y) + (b.x + b.y);
  xhi += 16.0f * ((c1.x + c1.y) + (c3.x + c3.y));
}

// Sum over the 16 lanes of each half warp (the 16 pieces of one 128-channel group).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int d = 8; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// One row of the gather, by one warp: x[p / top_k] scaled into f16 (permuted by
// perm_e when given, through the warp's shared-memory row buffer `stage`), or
// zeros for a padding row (p >= P).  With pg_corr the row is stored in the
// per-group-scaled layout above and its corrections go to pg_corr[g * cap + row].
template <bool BF16>
__device__ __forceinline__ void gather_one_row(const uint16_t* __restrict__ x, int p, int row, int P, int top_k, int H,
                                               int64_t cap, const int32_t* __restrict__ perm_e, uint4* stage,
                                               uint8_t* __restrict__ xg, float* __restrict__ xscale,
                                               float* __restrict__ pg_corr, int lane) {
  // Padding rows: zeros, except for batches of at most kNoPadPairs pairs, where
  // they are left as they are (a token row feeds only its own output column of
  // the GEMMs, an MMA column, and every epilogue drops the columns of padding
  // rows, pair >= P; measured on GB300: M = 1 layer 3 % faster, while at 32
  // pairs and more the GEMMs' reads of never-written rows cost 0.5-1.5 %).
  if (p >= P) {
    if (P <= kNoPadPairs) return;
    for (int c = lane; c < H / 8; c += 32)
      *reinterpret_cast<uint4*>(xg + staged_offset(row, 8 * c, cap)) = make_uint4(0, 0, 0, 0);
    if (lane == 0) xscale[row] = 1.0f;
    if (pg_corr != nullptr)
      for (int g = lane; g < H / 128; g += 32) pg_corr[g * cap + row] = 0.0f;
    return;
  }
  const uint16_t* src = x + static_cast<int64_t>(p / top_k) * H;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  // act-order: the row is staged in this warp's shared-memory buffer (coalesced
  // 16-byte loads) and permuted from there
  float amax = 0.0f;
  for (int i = lane; i < H / 8; i += 32) {
    const uint4 v = __ldg(s4 + i);
    if (perm_e != nullptr) stage[i] = v;
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(act_to_float<BF16>(e[k])));
  }
  amax = warp_max(amax);
  const float2 sc = row_exponent_scale(amax);
  const float inv = sc.y;
  if (lane == 0) xscale[row] = sc.x;
  if (perm_e != nullptr) __syncwarp();  // the staged row is complete
  const uint16_t* srow = reinterpret_cast<const uint16_t*>(stage);
  const int4* pr4 = reinterpret_cast<const int4*>(perm_e);
  // every lane runs every iteration (the per-group sums shuffle across the half warp)
  for (int c0 = 0; c0 < H / 8; c0 += 32) {
    const int c = c0 + lane;
    float xlo = 0.0f, xhi = 0.0f;
    if (c < H / 8) {
      uint16_t e[8];
      if (perm_e == nullptr) {
        *reinterpret_cast<uint4*>(e) = __ldg(s4 + c);
      } else {
        const int4 ka = __ldg(pr4 + 2 * c), kb = __ldg(pr4 + 2 * c + 1);
        e[0] = srow[ka.x]; e[1] = srow[ka.y]; e[2] = srow[ka.z]; e[3] = srow[ka.w];
        e[4] = srow[kb.x]; e[5] = srow[kb.y]; e[6] = srow[kb.z]; e[7] = srow[kb.w];
      }
      uint4 o = scale_to_f16x8<BF16>(e, inv);
      if (pg_corr != nullptr) pg_piece(o, xlo, xhi);
      *reinterpret_cast<uint4*>(xg + staged_offset(row, 8 * c, cap)) = o;
    }
    if (pg_corr != nullptr) {
      const float corr = half_warp_sum(1032.0f * xlo + 72.0f * xhi);
      const int g = (c0 >> 4) + (lane >> 4);  // the group of this half warp's 16 pieces
      if ((lane & 15) == 0 && c < H / 8) pg_corr[g * cap + row] = corr;
    }
  }
  if (perm_e != nullptr) __syncwarp();  // before the next row overwrites the buffer
}

template <bool BF16>
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_ids,
                  const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ num_post_padded,
                  const int32_t* __restrict__ perm13, int32_t P, int32_t top_k, int32_t H, int32_t B, int64_t cap,
                  uint8_t* __restrict__ xg, float* __restrict__ xscale, float* __restrict__ pg_corr) {
  extern __shared__ uint4 row_buf[];  // act-order only: one token row per warp
  pdl_launch_dependents();
  pdl_wait();
  const int total = *num_post_padded;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;  // warps (rows in flight) per block
  const int warps = gridDim.x * wpb;
  uint4* stage = perm13 != nullptr ? row_buf + (threadIdx.x >> 5) * (H / 8) : nullptr;
  for (int row = blockIdx.x * wpb + (threadIdx.x >> 5); row < total; row += warps) {
    const int32_t* perm_e = perm13 != nullptr ? perm13 + static_cast<int64_t>(expert_ids[row / B]) * H : nullptr;
    gather_one_row<BF16>(x, sorted_ids[row], row, P, top_k, H, cap, perm_e, stage, xg, xscale, pg_corr, lane);
  }
}

// ---------------------------------------------------------------------------
// moe_align and the token gather in one kernel, for small batches (P pairs at
// most kSmallPairs).  Every block groups the pairs itself in shared memory (the
// same result as moe_align_kernel: experts ascending, pairs ascending inside an
// expert, padding and tail = P, chunks of the token tile), block 0 publishes
// the grouping for the GEMMs, and each block then gathers its rows.  This takes
// one kernel boundary off the critical path of decode-sized batches.
// ---------------------------------------------------------------------------
constexpr int kSmallPairs = 1024;

// Exclusive scan of one value per thread over a block of kGatherThreads threads.
__device__ __forceinline__ int block_exclusive_scan_256(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kW = kGatherThreads / 32;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kW ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < kW; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    if (lane < kW) warp_sums[lane] = w;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = warp_sums[kW - 1];
  __syncthreads();
  return excl;
}

template <bool BF16>
__global__ void __launch_bounds__(kGatherThreads)
    align_gather_small_kernel(const int32_t* __restrict__ ids, int32_t P, int32_t E, int32_t B, int64_t capacity,
                              int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                              int32_t* __restrict__ num_post_padded, int32_t T, Chunk* __restrict__ chunks,
                              int32_t* __restrict__ n_chunks, int32_t* __restrict__ status,
                              const uint16_t* __restrict__ x, const int32_t* __restrict__ perm13, int32_t top_k,
                              int32_t H, int64_t cap, uint8_t* __restrict__ xg, float* __restrict__ xscale,
                              float* __restrict__ pg_corr) {
  extern __shared__ __align__(16) int32_t sm_i[];
  __shared__ int warp_sums[kGatherThreads / 32];
  __shared__ int s_bad;
  const int rows_max = P + E * (B - 1);
  int32_t* s_ids = sm_i;                 // [P]
  int32_t* s_cnt = s_ids + P;            // [E] pair counts
  int32_t* s_off = s_cnt + E;            // [E] first row of each expert
  int32_t* s_cur = s_off + E;            // [E] scatter cursors
  int32_t* s_sorted = s_cur + E;         // [rows_max]
  // act-order row buffers (uint4): 16-byte aligned after the integer arrays
  uint4* stage_base = reinterpret_cast<uint4*>(sm_i + ((P + 3 * E + rows_max + 3) & ~3));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel in the stream has completed (no-op without PDL)

  if (tid == 0) s_bad = 0;
  for (int i = tid; i < E; i += kGatherThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int i = tid; i < P; i += kGatherThreads) {
    const int e = ids != nullptr ? __ldg(ids + i) : 0;  // no ids: every pair is expert 0
    s_ids[i] = e;
    if (e >= 0 && e < E)
      atomicAdd(s_cnt + e, 1);
    else
      s_bad = 1;
  }
  __syncthreads();
  // padded sizes, offsets and chunk counts: thread t owns experts [t*per, (t+1)*per)
  const int per = (E + kGatherThreads - 1) / kGatherThreads;
  const int e0 = tid * per, e1 = min(E, e0 + per);
  int pad_sum = 0, nch_sum = 0;
  for (int e = e0; e < e1; ++e) {
    const int pad = (s_cnt[e] + B - 1) / B * B;
    pad_sum += pad;
    nch_sum += (T > 0) ? (pad + T - 1) / T : 0;
  }
  int total, total_chunks;
  int run = block_exclusive_scan_256(pad_sum, warp_sums, &total);
  int crun = block_exclusive_scan_256(nch_sum, warp_sums, &total_chunks);
  for (int e = e0; e < e1; ++e) {
    const int cnt = s_cnt[e];
    const int pad = (cnt + B - 1) / B * B;
    s_off[e] = run;
    s_cur[e] = run;
    for (int i = run + cnt; i < run + pad; ++i) s_sorted[i] = P;  // padding rows of expert e
    if (blockIdx.x == 0) {
      for (int b = run / B; b < (run + pad) / B; ++b) expert_ids[b] = e;
      const int nch = (T > 0) ? (pad + T - 1) / T : 0;
      for (int c = 0; c < nch; ++c) {
        Chunk ch;
        ch.expert = e;
        ch.row0 = run + c * T;
        ch.nrows = min(T, pad - c * T);
        ch.first = crun;
        ch.count = nch;
        ch.pad = 0;
        chunks[crun + c] = ch;
      }
      crun += nch;
    }
    run += pad;
  }
  __syncthreads();
  // stable scatter: one warp walks the pairs in order, grouping lanes by expert
  if (warp == 0) {
    for (int base = 0; base < P; base += 32) {
      const int p = base + lane;
      const int e = p < P ? s_ids[p] : -1;
      const bool valid = e >= 0 && e < E;
      const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
      if (valid) s_sorted[s_cur[e] + __popc(peers & ((1u << lane) - 1u))] = p;
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) s_cur[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int64_t i = tid; i < capacity; i += kGatherThreads) sorted_ids[i] = i < total ? s_sorted[i] : P;
    const int64_t nblocks = (capacity + B - 1) / B;
    for (int64_t b = total / B + tid; b < nblocks; b += kGatherThreads) expert_ids[b] = -1;
    if (tid == 0) {
      *num_post_padded = total;
      if (n_chunks != nullptr) *n_chunks = total_chunks;
      if (status != nullptr) *status = s_bad ? kStatusBadExpert : 0;
    }
  }
  // the gather of this block's rows
  uint4* stage = perm13 != nullptr ? stage_base + warp * (H / 8) : nullptr;
  const int wpb = kGatherThreads / 32;
  for (int row = blockIdx.x * wpb + warp; row < total; row += gridDim.x * wpb) {
    const int32_t* perm_e = nullptr;
    if (perm13 != nullptr) {
      // the expert whose rows [s_off[e], s_off[e] + padded) hold this row: the last e with
      // s_off[e] <= row (an empty expert shares its offset with the next one, which comes later)
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= row) lo = mid; else hi = mid - 1;
      }
      perm_e = perm13 + static_cast<int64_t>(lo) * H;
    }
    gather_one_row<BF16>(x, s_sorted[row], row, P, top_k, H, cap, perm_e, stage, xg, xscale, pg_corr, lane);
  }
}

cudaError_t launch_gather(const void* x, bool bf16, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* num_post_padded, const int32_t* perm13, int32_t P, int32_t top_k,
                          int32_t H, int32_t block, int64_t cap_rows, void* xg, float* xscale, float* pg_corr,
                          int num_sms, cudaStream_t stream) {
  // act-order: each warp stages its token row in shared memory (H x 2 bytes per
  // warp, at most 8 warps and about 200 KB per block)
  int wpb = kGatherThreads / 32;
  if (perm13 != nullptr) wpb = std::max(1, std::min(wpb, static_cast<int>((200 * 1024) / (2 * static_cast<int64_t>(H)))));
  const int64_t want = (cap_rows + wpb - 1) / wpb;
  const int grid = static_cast<int>(want < 4LL * num_sms ? (want > 0 ? want : 1) : 4LL * num_sms);
  auto kern = bf16 ? gather_kernel<true> : gather_kernel<false>;
  const size_t smem = perm13 != nullptr ? static_cast<size_t>(wpb) * H * 2 : 0;
  if (smem > 48 * 1024) {
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  return launch_kernel(kern, dim3(grid), dim3(32 * wpb), smem, stream, true, static_cast<const uint16_t*>(x),
                       sorted_ids, expert_ids, num_post_padded, perm13, P, top_k, H, block, cap_rows,
                       static_cast<uint8_t*>(xg), xscale, pg_corr);
}

// ---------------------------------------------------------------------------
// Split-K gate/up reduce: inter32[row, j] = SiLU(sum_s h[s, row, 2j]) * sum_s h[s, row, 2j+1]
// (the packed gate/up GEMM interleaves gate and up rows, so h is [.., g0, u0, g1, u1, ..]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__global__ void __launch_bounds__(256)
    silu_reduce_kernel(const float* __restrict__ h, const int32_t* __restrict__ num_post_padded, int32_t split,
                       int64_t cap_rows, int32_t I, float* __restrict__ inter32) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = static_cast<int64_t>(*num_post_padded) * (I / 2);  // two j per thread
  const int64_t slab = cap_rows * 2 * static_cast<int64_t>(I);
  for (int64_t t = blockIdx.x * 256LL + threadIdx.x; t < total; t += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t row = t / (I / 2);
    const int j2 = static_cast<int>(t - row * (I / 2));
    const int64_t base = row * 2 * I + 4LL * j2;
    float4 acc = __ldg(reinterpret_cast<const float4*>(h + base));
    for (int s = 1; s < split; ++s) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(h + s * slab + base));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float2*>(inter32 + row * I)[j2] = make_float2(silu_f(acc.x) * acc.y, silu_f(acc.z) * acc.w);
  }
}

size_t align_gather_small_smem(int32_t P, int32_t E, int32_t block, int32_t H, bool act_order) {
  const int64_t rows_max = static_cast<int64_t>(P) + static_cast<int64_t>(E) * (block - 1);
  // the integer arrays, rounded up to 16 bytes where the row buffers start
  const size_t ints = (static_cast<size_t>(P) + 3 * static_cast<size_t>(E) + static_cast<size_t>(rows_max) + 3) & ~size_t(3);
  return ints * 4 + (act_order ? static_cast<size_t>(kGatherThreads / 32) * H * 2 : 0);
}

bool align_gather_small_fits(int32_t P, int32_t E, int32_t block, int32_t H, bool act_order) {
  return P <= kSmallPairs && align_gather_small_smem(P, E, block, H, act_order) <= 200 * 1024;
}

cudaError_t launch_align_gather_small(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block, int64_t capacity,
                                      int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                                      int32_t token_tile, Chunk* chunks, int32_t* n_chunks, int32_t* status,
                                      const void* x, bool bf16, const int32_t* perm13, int32_t top_k, int32_t H,
                                      int64_t cap_rows, void* xg, float* xscale, float* pg_corr, int num_sms,
                                      cudaStream_t stream) {
  const size_t smem = align_gather_small_smem(P, E, block, H, perm13 != nullptr);
  const int wpb = kGatherThreads / 32;
  const int64_t want = (cap_rows + wpb - 1) / wpb;
  const int grid = static_cast<int>(want < 4LL * num_sms ? (want > 0 ? want : 1) : 4LL * num_sms);
  auto kern = bf16 ? align_gather_small_kernel<true> : align_gather_small_kernel<false>;
  if (smem > 48 * 1024) {
    const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  // First kernel of a forward.  Up to 64 pairs it is launched as a programmatic
  // dependent: it waits (griddepcontrol.wait) for the previous kernel in the
  // stream before it reads or writes anything, and its launch overlaps that
  // kernel's tail (a kernel that never signals behaves as plain stream order).
  // Measured on GB300: Mixtral int4 M = 1 layer -2.5 %, dense linear M = 1/16
  // -4 %; at 128 pairs and more the early CTAs cost 6-7 %.
  const bool pdl = P <= 64;
  return launch_kernel(kern, dim3(grid), dim3(kGatherThreads), smem, stream, pdl, topk_ids, P, E, block, capacity,
                       sorted_ids, expert_ids, num_post_padded, token_tile, chunks, n_chunks, status,
                       static_cast<const uint16_t*>(x), perm13, top_k, H, cap_rows, static_cast<uint8_t*>(xg), xscale,
                       pg_corr);
}

cudaError_t launch_silu_reduce(const float* h, const int32_t* num_post_padded, int32_t split, int64_t cap_rows,
                               int32_t I, float* inter32, int num_sms, cudaStream_t stream) {
  return launch_kernel(silu_reduce_kernel, dim3(4 * num_sms), dim3(256), 0, stream, true, h, num_post_padded, split,
                       cap_rows, I, inter32);
}

// ---------------------------------------------------------------------------
// Intermediate rescale: row `row` of the down GEMM's B operand is
// inter32[row, :] * 2^-e_row in f16 in the pre-staged layout (staged_offset),
// iscale[row] = 2^e_row.  One CTA per row (the absmax is a block reduction);
// padding rows get zeros and scale 1 without reading inter32 (left as they are
// for batches of at most kNoPadPairs pairs, see gather_one_row).
// ---------------------------------------------------------------------------
constexpr int kRescaleThreads = 256;

__global__ void __launch_bounds__(kRescaleThreads)
    inter_rescale_kernel(const float* __restrict__ inter32, const int32_t* __restrict__ num_post_padded,
                         const int32_t* __restrict__ sorted_ids, int32_t P, int32_t I, int64_t cap,
                         uint8_t* __restrict__ inter16, float* __restrict__ iscale, float* __restrict__ pg_corr,
                         const TopkPrep prep) {
  __shared__ float red[kRescaleThreads / 32];
  pdl_launch_dependents();
  pdl_wait();
  if (prep.cnt != nullptr) {
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRescaleThreads + threadIdx.x;
    const int64_t ts = static_cast<int64_t>(gridDim.x) * kRescaleThreads;
    for (int64_t i = t0; i < prep.n_cnt; i += ts) prep.cnt[i] = 0;
    for (int64_t m = t0; m < prep.M; m += ts) {
      bool any = false;
      for (int j = 0; j < prep.top_k; ++j) {
        const int e = prep.topk_ids[m * prep.top_k + j];
        any = any || (e >= 0 && e < prep.E);
      }
      if (!any)
        for (int n = 0; n < prep.H; ++n) prep.out[m * prep.H + n] = 0;
    }
  }
  const int total = *num_post_padded;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int row = blockIdx.x; row < total; row += gridDim.x) {
    if (sorted_ids[row] >= P) {  // padding row (uniform across the CTA), see gather_one_row
      if (P <= kNoPadPairs) continue;
      for (int c = threadIdx.x; c < I / 8; c += kRescaleThreads)
        *reinterpret_cast<uint4*>(inter16 + staged_offset(row, 8 * c, cap)) = make_uint4(0, 0, 0, 0);
      if (threadIdx.x == 0) iscale[row] = 1.0f;
      if (pg_corr != nullptr)
        for (int g = threadIdx.x; g < I / 128; g += kRescaleThreads) pg_corr[g * cap + row] = 0.0f;
      continue;
    }
    const float4* s4 = reinterpret_cast<const float4*>(inter32 + static_cast<int64_t>(row) * I);
    float amax = 0.0f;
    for (int i = threadIdx.x; i < I / 4; i += kRescaleThreads) {
      const float4 v = __ldg(s4 + i);
      amax = fmaxf(fmaxf(fmaxf(amax, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
    }
    amax = warp_max(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < kRescaleThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();  // red is reused by the next row
    const float2 sc = row_exponent_scale(amax);
    if (threadIdx.x == 0) iscale[row] = sc.x;
    // every thread runs every iteration (the per-group sums shuffle across half warps)
    for (int c0 = 0; c0 < I / 8; c0 += kRescaleThreads) {
      const int c = c0 + threadIdx.x;
      float xlo = 0.0f, xhi = 0.0f;
      if (c < I / 8) {
        const float4 a = __ldg(s4 + 2 * c), b = __ldg(s4 + 2 * c + 1);
        uint4 o;
        o.x = static_cast<uint32_t>(f16_bits(a.x * sc.y)) | (static_cast<uint32_t>(f16_bits(a.y * sc.y)) << 16);
        o.y = static_cast<uint32_t>(f16_bits(a.z * sc.y)) | (static_cast<uint32_t>(f16_bits(a.w * sc.y)) << 16);
        o.z = static_cast<uint32_t>(f16_bits(b.x * sc.y)) | (static_cast<uint32_t>(f16_bits(b.y * sc.y)) << 16);
        o.w = static_cast<uint32_t>(f16_bits(b.z * sc.y)) | (static_cast<uint32_t>(f16_bits(b.w * sc.y)) << 16);
        if (pg_corr != nullptr) pg_piece(o, xlo, xhi);
        *reinterpret_cast<uint4*>(inter16 + staged_offset(row, 8 * c, cap)) = o;
      }
      if (pg_corr != nullptr) {
        const float corr = half_warp_sum(1032.0f * xlo + 72.0f * xhi);
        if ((threadIdx.x & 15) == 0 && c < I / 8) pg_corr[(c >> 4) * cap + row] = corr;
      }
    }
  }
}

cudaError_t launch_inter_rescale(const float* inter32, const int32_t* num_post_padded, const int32_t* sorted_ids,
                                 int32_t P, int32_t I, int64_t cap_rows, void* inter16, float* iscale, float* pg_corr,
                                 const TopkPrep& prep, int num_sms, cudaStream_t stream) {
  const int grid = static_cast<int>(cap_rows < 8LL * num_sms ? (cap_rows > 0 ? cap_rows : 1) : 8LL * num_sms);
  return launch_kernel(inter_rescale_kernel, dim3(grid), dim3(kRescaleThreads), 0, stream, true, inter32,
                       num_post_padded, sorted_ids, P, I, cap_rows, static_cast<uint8_t*>(inter16), iscale, pg_corr,
                       prep);
}

// ---------------------------------------------------------------------------
// Output reduce: out[m, n] = sum_j sum_s y[s, m*top_k + j, n] in a fixed order
// (the routing weight is already applied by the down GEMM's epilogue).  Slots
// whose expert id is outside [0, E) were dropped by moe_align, so no GEMM wrote
// their y rows: they are skipped.
// ---------------------------------------------------------------------------
template <bool BF16>
__global__ void __launch_bounds__(256)
    out_reduce_kernel(const float* __restrict__ y, const int32_t* __restrict__ topk_ids, int32_t E, int32_t split,
                      int64_t M, int32_t top_k, int32_t H, uint16_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = M * (H / 4);
  const int64_t slab = M * top_k * static_cast<int64_t>(H);
  for (int64_t t = blockIdx.x * 256LL + threadIdx.x; t < total; t += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t m = t / (H / 4);
    const int n4 = static_cast<int>(t - m * (H / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < top_k; ++j) {
      const int e = __ldg(topk_ids + m * top_k + j);
      if (e < 0 || e >= E) continue;
      const int64_t base = (m * top_k + j) * H + 4LL * n4;
      for (int s = 0; s < split; ++s) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(y + s * slab + base));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
    }
    uint2 packed;
    if (BF16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
      packed.x = *reinterpret_cast<uint32_t*>(&a);
      packed.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 a = __floats2half2_rn(acc.x, acc.y), b = __floats2half2_rn(acc.z, acc.w);
      packed.x = *reinterpret_cast<uint32_t*>(&a);
      packed.y = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint2*>(out + m * H)[n4] = packed;
  }
}

cudaError_t launch_out_reduce(const float* y, const int32_t* topk_ids, int32_t E, int32_t split, int64_t M,
                              int32_t top_k, int32_t H, bool bf16, void* out, int num_sms, cudaStream_t stream) {
  const int64_t want = (M * (H / 4) + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
  if (bf16)
    return launch_kernel(out_reduce_kernel<true>, dim3(grid), dim3(256), 0, stream, true, y, topk_ids, E, split, M,
                         top_k, H, static_cast<uint16_t*>(out));
  return launch_kernel(out_reduce_kernel<false>, dim3(grid), dim3(256), 0, stream, true, y, topk_ids, E, split, M,
                       top_k, H, static_cast<uint16_t*>(out));
}

// ---------------------------------------------------------------------------
// Dense linear, split K: out[m, n] = sum_s h[s, m, n] in a fixed order, cast to
// the activation type (the GEMM's epilogue applied every scale).
// ---------------------------------------------------------------------------
template <bool BF16>
__global__ void __launch_bounds__(256)
    linear_reduce_kernel(const float* __restrict__ h, int32_t split, int64_t cap_rows, int64_t M, int32_t N,
                         uint16_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = M * (N / 4);
  const int64_t slab = cap_rows * static_cast<int64_t>(N);
  for (int64_t t = blockIdx.x * 256LL + threadIdx.x; t < total; t += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t m = t / (N / 4);
    const int n4 = static_cast<int>(t - m * (N / 4));
    const int64_t base = m * N + 4LL * n4;
    float4 acc = __ldg(reinterpret_cast<const float4*>(h + base));
    for (int s = 1; s < split; ++s) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(h + s * slab + base));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    uint2 packed;
    if (BF16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
      packed.x = *reinterpret_cast<uint32_t*>(&a);
      packed.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 a = __floats2half2_rn(acc.x, acc.y), b = __floats2half2_rn(acc.z, acc.w);
      packed.x = *reinterpret_cast<uint32_t*>(&a);
      packed.y = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint2*>(out + m * N)[n4] = packed;
  }
}

cudaError_t launch_linear_reduce(const float* h, int32_t split, int64_t cap_rows, int64_t M, int32_t N, bool bf16,
                                 void* out, int num_sms, cudaStream_t stream) {
  const int64_t want = (M * (N / 4) + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
  if (bf16)
    return launch_kernel(linear_reduce_kernel<true>, dim3(grid), dim3(256), 0, stream, true, h, split, cap_rows, M,
                         N, static_cast<uint16_t*>(out));
  return launch_kernel(linear_reduce_kernel<false>, dim3(grid), dim3(256), 0, stream, true, h, split, cap_rows, M, N,
                       static_cast<uint16_t*>(out));
}

// ---------------------------------------------------------------------------
// Router: per token row, the top-k experts by logit (ties go to the lower
// expert id) in rank order and their softmax probabilities, renormalised over
// the kept experts when asked.  One warp per row; lane l holds the logits of
// experts l, l+32, ... (E <= 1024) in registers; k rounds of a warp arg-max.
// NaN logits count as -inf.
// ---------------------------------------------------------------------------
constexpr int kRouteThreads = 256;

template <int DT>  // 0: f32, 1: f16, 2: bf16
__device__ __forceinline__ float load_logit(const void* base, int64_t i) {
  float v;
  if (DT == 0) {
    v = __ldg(static_cast<const float*>(base) + i);
  } else {
    const uint16_t b = __ldg(static_cast<const uint16_t*>(base) + i);
    v = (DT == 1) ? __half2float(__ushort_as_half(b)) : __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  return (v != v) ? -INFINITY : v;
}

template <int DT>
__global__ void __launch_bounds__(kRouteThreads)
    route_topk_kernel(const void* __restrict__ logits, int64_t M, int32_t E, int32_t k, int32_t renormalize,
                      int32_t* __restrict__ topk_ids, float* __restrict__ topk_weights) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRouteThreads / 32);
  for (int64_t m = blockIdx.x * static_cast<int64_t>(kRouteThreads / 32) + (threadIdx.x >> 5); m < M; m += warps) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = lane + 32 * j;
      v[j] = (e < E) ? load_logit<DT>(logits, m * E + e) : -INFINITY;
    }
    uint32_t taken = 0;
    float my_v = -INFINITY;
    int my_e = 0;
    for (int r = 0; r < k; ++r) {
      float best = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && (v[j] > best || (v[j] == best && e < be))) {
          best = v[j];
          be = e;
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, d);
        const int oe = __shfl_xor_sync(0xffffffffu, be, d);
        if (ov > best || (ov == best && oe < be)) {
          best = ov;
          be = oe;
        }
      }
      if (lane == (be & 31)) taken |= 1u << (be >> 5);
      if (lane == r) {
        my_v = best;
        my_e = be;
      }
    }
    // the first kept logit is the row maximum; a row of -inf logits routes uniformly
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    const bool masked = top == -INFINITY;
    const float pk = (lane < k) ? (masked ? 1.0f : expf(my_v - top)) : 0.0f;
    float denom = 0.0f;
    if (renormalize) {
      denom = pk;
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (lane + 32 * j < E) denom += masked ? 1.0f : expf(v[j] - top);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, d);
    if (lane < k) {
      topk_ids[m * k + lane] = my_e;
      topk_weights[m * k + lane] = pk / denom;
    }
  }
}

cudaError_t launch_route_topk(const void* logits, int dtype, int64_t M, int32_t E, int32_t k, int32_t renormalize,
                              int32_t* topk_ids, float* topk_weights, int num_sms, cudaStream_t stream) {
  const int64_t want = (M + (kRouteThreads / 32) - 1) / (kRouteThreads / 32);
  const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
  auto kern = dtype == 0 ? route_topk_kernel<0> : dtype == 1 ? route_topk_kernel<1> : route_topk_kernel<2>;
  return launch_kernel(kern, dim3(grid), dim3(kRouteThreads), 0, stream, false, logits, M, E, k, renormalize,
                       topk_ids, topk_weights);
}

}  // namespace qmoe
