// aux_kernels.cu - the non-GEMM steps of the fused MoE layer on sm_103a:
//   moe_align_block_size  (group token-expert pairs by expert, pad to the block)
//   token gather          (sorted, padded, act-order-permuted activation rows)
//   split-K SiLU reduce   (sum gate/up partials, apply SiLU(gate)*up)
//   output reduce         (sum the top-k weighted expert outputs per token)
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
  pdl_wait();  // no-op unless launched as a dependent

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
    const int e = in ? __ldg(ids + p) : -1;
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
    const int ex = in ? __ldg(ids + p) : -1;
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
  // first kernel of a forward: ordinary stream order behind the caller's work
  return launch_kernel(moe_align_kernel, dim3(1), dim3(kAlignThreads), smem, stream, false, topk_ids, P, E, block,
                       capacity, sorted_ids, expert_ids, num_post_padded, chunks ? token_tile : 0, chunks, n_chunks,
                       status);
}

// ---------------------------------------------------------------------------
// Token gather: xg[row, :] = x[sorted_ids[row] / top_k, perm13_e] (zeros for
// padding rows).  Rows are the B operand of the gate/up GEMM; with act-order
// the hidden channels are put in each expert's sorted-group order so the GEMM
// walks K in whole quantization groups.
// ---------------------------------------------------------------------------
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_ids,
                  const int32_t* __restrict__ expert_ids, const int32_t* __restrict__ num_post_padded,
                  const int32_t* __restrict__ perm13, int32_t P, int32_t top_k, int32_t H, int32_t B,
                  uint16_t* __restrict__ xg) {
  pdl_launch_dependents();
  pdl_wait();
  const int total = *num_post_padded;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kGatherThreads / 32);
  for (int row = blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); row < total; row += warps) {
    const int p = sorted_ids[row];
    uint16_t* dst = xg + static_cast<int64_t>(row) * H;
    if (p >= P) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int i = lane; i < H / 8; i += 32) d4[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint16_t* src = x + static_cast<int64_t>(p / top_k) * H;
    if (perm13 == nullptr) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int i = lane; i < H / 8; i += 32) d4[i] = __ldg(s4 + i);
    } else {
      const int32_t* pr = perm13 + static_cast<int64_t>(expert_ids[row / B]) * H;
      uint32_t* d2 = reinterpret_cast<uint32_t*>(dst);
      for (int i = lane; i < H / 2; i += 32) {
        const int2 k2 = __ldg(reinterpret_cast<const int2*>(pr) + i);
        d2[i] = static_cast<uint32_t>(__ldg(src + k2.x)) | (static_cast<uint32_t>(__ldg(src + k2.y)) << 16);
      }
    }
  }
}

cudaError_t launch_gather(const void* x, const int32_t* sorted_ids, const int32_t* expert_ids,
                          const int32_t* num_post_padded, const int32_t* perm13, int32_t P, int32_t top_k,
                          int32_t H, int32_t block, int64_t cap_rows, void* xg, int num_sms, cudaStream_t stream) {
  const int64_t want = (cap_rows + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
  const int grid = static_cast<int>(want < 4LL * num_sms ? (want > 0 ? want : 1) : 4LL * num_sms);
  return launch_kernel(gather_kernel, dim3(grid), dim3(kGatherThreads), 0, stream, true,
                       static_cast<const uint16_t*>(x), sorted_ids, expert_ids, num_post_padded, perm13, P, top_k, H,
                       block, static_cast<uint16_t*>(xg));
}

// ---------------------------------------------------------------------------
// Split-K gate/up reduce: inter[row, j] = SiLU(sum_s h[s, row, 2j]) * sum_s h[s, row, 2j+1]
// (the packed gate/up GEMM interleaves gate and up rows, so h is [.., g0, u0, g1, u1, ..]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <bool BF16>
__global__ void __launch_bounds__(256)
    silu_reduce_kernel(const float* __restrict__ h, const int32_t* __restrict__ num_post_padded, int32_t split,
                       int64_t cap_rows, int32_t I, uint16_t* __restrict__ inter, int64_t lo_offset) {
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
    const float r0 = silu_f(acc.x) * acc.y;
    const float r1 = silu_f(acc.z) * acc.w;
    uint32_t packed, packed_lo = 0;
    if (BF16) {
      __nv_bfloat162 b = __floats2bfloat162_rn(r0, r1);
      packed = *reinterpret_cast<uint32_t*>(&b);
      // second bf16 term carries the rounding residual of the first
      __nv_bfloat162 l = __floats2bfloat162_rn(r0 - __bfloat162float(b.x), r1 - __bfloat162float(b.y));
      packed_lo = *reinterpret_cast<uint32_t*>(&l);
    } else {
      __half2 b = __floats2half2_rn(r0, r1);
      packed = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint32_t*>(inter + row * I)[j2] = packed;
    if (lo_offset != 0) reinterpret_cast<uint32_t*>(inter + lo_offset + row * I)[j2] = packed_lo;
  }
}

cudaError_t launch_silu_reduce(const float* h, const int32_t* num_post_padded, int32_t split, int64_t cap_rows,
                               int32_t I, bool bf16, void* inter, int64_t inter_lo_offset, int num_sms,
                               cudaStream_t stream) {
  const int grid = 4 * num_sms;
  if (bf16)
    return launch_kernel(silu_reduce_kernel<true>, dim3(grid), dim3(256), 0, stream, true, h, num_post_padded, split,
                         cap_rows, I, static_cast<uint16_t*>(inter), inter_lo_offset);
  return launch_kernel(silu_reduce_kernel<false>, dim3(grid), dim3(256), 0, stream, true, h, num_post_padded, split,
                       cap_rows, I, static_cast<uint16_t*>(inter), int64_t(0));
}

// ---------------------------------------------------------------------------
// Output reduce: out[m, n] = sum_j sum_s y[s, m*top_k + j, n] in a fixed order
// (the routing weight is already applied by the down GEMM's epilogue).
// ---------------------------------------------------------------------------
template <bool BF16>
__global__ void __launch_bounds__(256)
    out_reduce_kernel(const float* __restrict__ y, int32_t split, int64_t M, int32_t top_k, int32_t H,
                      uint16_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = M * (H / 4);
  const int64_t slab = M * top_k * static_cast<int64_t>(H);
  for (int64_t t = blockIdx.x * 256LL + threadIdx.x; t < total; t += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t m = t / (H / 4);
    const int n4 = static_cast<int>(t - m * (H / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < top_k; ++j) {
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

cudaError_t launch_out_reduce(const float* y, int32_t split, int64_t M, int32_t top_k, int32_t H, bool bf16,
                              void* out, int num_sms, cudaStream_t stream) {
  const int64_t want = (M * (H / 4) + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * num_sms ? (want > 0 ? want : 1) : 8LL * num_sms);
  if (bf16)
    return launch_kernel(out_reduce_kernel<true>, dim3(grid), dim3(256), 0, stream, true, y, split, M, top_k, H,
                         static_cast<uint16_t*>(out));
  return launch_kernel(out_reduce_kernel<false>, dim3(grid), dim3(256), 0, stream, true, y, split, M, top_k, H,
                       static_cast<uint16_t*>(out));
}

}  // namespace qmoe
