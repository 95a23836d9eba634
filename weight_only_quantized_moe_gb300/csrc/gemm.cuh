// gemm.cuh - grouped expert GEMM with on-the-fly weight dequantization for sm_103a.
//
// What it computes (pages "Marlin moe integration" and "[Kernel] W8A16 Int8
// inside FusedMoE": the fused MoE kernel consumes already-quantized expert
// weights and casts them to FP16/BF16 inside the kernel before the matmul):
// for one expert e, a tile of 128 output features and a chunk of token rows,
//     acc[f, t] = sum_k W_e[f, k] * B[t, k]
// where W_e is dequantized from packed int4 (with its group scale) or int8,
// and B is the chunk's rows of the gathered activations (gate/up GEMM) or of
// the intermediate (down GEMM).  The epilogue then applies SiLU(gate)*up, or
// the routing weight, per the mode.
//
// Numerics: both operands are f16 whatever the activation type.  B rows are
// stored scaled by a power of two per row (exact, see aux_kernels.cu) and the
// epilogue multiplies each accumulator column back; int4 weights (q - 8) * s
// are exact in f16 when s is a bf16 scale (3 + 8 significant bits) and rounded
// once when s is an f16 scale; int8 codes are exact and their per-row scale is
// applied to the fp32 accumulator.
//
// Design for GB300 (prior-art Marlin/Triton kernels staged both operands in
// shared memory; here only the tokens are):
//   * swap-AB: the 128 weight rows are the MMA's M; the chunk's token rows
//     (16..128) are N, so tiny decode batches waste no tensor work.
//   * the dequantized weight tile goes registers -> TMEM (tcgen05.st) and is
//     the MMA's A operand straight from tensor memory; dequantized weights
//     never touch shared memory, which carries only the packed bytes and the
//     token tile.
//   * a pipeline stage covers `ks` (1 or 2) quantization groups of 128 K.  Its
//     packed weights (contiguous blocks per 128x128 tile, scales appended) and
//     its token tile arrive as two 1-D bulk TMA copies: the producers of the
//     B operand (gather, rescale) store it pre-staged, per stage and 8-row
//     group, in the 128-byte-swizzled K-major layout the MMA's shared-memory
//     descriptor reads, so a chunk's tile for one stage is one contiguous run.
//   * warp roles: two TMA producer threads (warps 4, 7), two MMA-issuing
//     threads (warps 5, 6) and two dequant warpgroups (warps 8-15), each pair
//     taking the even and the odd pipeline stages; one epilogue warpgroup
//     (warps 0-3) reads the fp32 accumulators out of TMEM.  Issuing a stage's
//     copies or MMAs costs one thread several hundred cycles, so the stage
//     rate at decode sizes needs two issuers of each.  A persistent grid walks
//     the work items.
//   * every mbarrier wait is bounded (see ptx.cuh); a wait that gives up
//     records QMOE_ERR_TIMEOUT in the status word and the CTA winds down after
//     waiting for its own copies and MMAs, then frees its TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qmoe_internal.h"

namespace qmoe {

constexpr int kGemmThreads = 512;
constexpr int kProducerWarp = 4;
constexpr int kProducerWarp2 = 7;
constexpr int kMmaWarp = 5;
constexpr int kDequantWarp0 = 8;  // warps 8..15: two warpgroups
constexpr uint32_t kTmemCols = 512;
constexpr int kBarrierBytes = 1024;

__host__ __device__ inline uint32_t gemm_w_region(int bytes) { return (bytes + 1023u) & ~1023u; }
// Shared memory of one pipeline stage: the token tile (T rows x ks*128 K x 2 B)
// then the packed weights of ks groups.
__host__ __device__ inline uint32_t gemm_stage_bytes(int token_tile, int group_bytes, int ks) {
  return static_cast<uint32_t>(token_tile) * 256u * ks + gemm_w_region(group_bytes * ks);
}

struct WorkItem {
  int e, row0, nrows, tile, split_idx, ks0, ks1;
};

// Work item i -> (split, chunk, tile).  Items of one split are rastered in
// groups of `chunk_group` chunks: tiles vary slowest inside a group so that the
// CTAs running at the same time share the group's token tiles and each expert
// weight tile in L2.
__device__ __forceinline__ void decode_item(const GemmParams& p, int nch, int i, WorkItem& w) {
  const int per_split = nch * p.n_tiles;
  const int s = i / per_split;
  const int r = i - s * per_split;
  const int grp_items = p.chunk_group * p.n_tiles;
  const int g = r / grp_items;
  const int rem = r - g * grp_items;
  const int c0 = g * p.chunk_group;
  const int cg = min(p.chunk_group, nch - c0);
  const int tile = rem / cg;
  const int c = c0 + (rem - tile * cg);
  const Chunk ch = p.chunks[c];
  w.e = ch.expert;
  w.row0 = ch.row0;
  w.nrows = ch.nrows;
  w.tile = tile;
  w.split_idx = s;
  const int k_units = p.k_groups / p.ks;
  w.ks0 = static_cast<int>(static_cast<int64_t>(k_units) * s / p.split);
  w.ks1 = static_cast<int>(static_cast<int64_t>(k_units) * (s + 1) / p.split);
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int32_t* status) {
  *abort_flag = 1;
  if (status != nullptr) atomicCAS(status, 0, kStatusTimeout);
}

// Wait that only gives up on the time limit (used while draining in-flight work).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const int never = 0;
  return mbar_wait(bar, parity, &never);
}

// ---------------------------------------------------------------------------
// Dequantization of one 128-K stage of one weight row into 64 TMEM columns
// (column c holds K elements 2c (low half) and 2c+1 (high half)), as f16.
// ---------------------------------------------------------------------------
// int4: packed chunk c (16 bytes) of the row holds K = 32c .. 32c+31; in word j
// of the chunk, nibble i holds K = 32c+8j+2i and nibble i+4 holds K = 32c+8j+2i+1.
// Magic-number conversion: (nibble | 0x6400) is the f16 value 1024 + q, exact,
// and subtracting 1032 gives q - 8 exactly; nibbles i = 1, 3 stay in bits 4..7
// of their half, where (nibble << 4) | 0x6400 is 1024 + 16q and
// fma(v, 1/16, -72) = q - 8 exactly, so one shift per word serves i = 2, 3.
// One multiply by the group scale rounds once (exact for bf16 scales).
template <bool BF16S>
__device__ __forceinline__ void dequant_int4_row(const uint4 (&pk)[4], uint32_t sbits, uint32_t (&out)[64]) {
  const uint32_t bias_bits = 0x64086408u;                        // 1032
  const uint32_t sixteenth = 0x2C002C00u, m72 = 0xD480D480u;     // 1/16, -72
  uint16_t s16;
  if (BF16S) {
    const __half h = __float2half_rn(__uint_as_float(sbits << 16));
    s16 = *reinterpret_cast<const uint16_t*>(&h);
  } else {
    s16 = static_cast<uint16_t>(sbits);
  }
  const uint32_t s2bits = static_cast<uint32_t>(s16) | (static_cast<uint32_t>(s16) << 16);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {pk[c].x, pk[c].y, pk[c].z, pk[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t src[2] = {w[j], w[j] >> 8};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lo = (src[h] & 0x000F000Fu) | 0x64006400u;
        const uint32_t hi = (src[h] & 0x00F000F0u) | 0x64006400u;
        __half2 vl = __hsub2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&bias_bits));
        __half2 vh = __hfma2(*reinterpret_cast<const __half2*>(&hi), *reinterpret_cast<const __half2*>(&sixteenth),
                             *reinterpret_cast<const __half2*>(&m72));
        vl = __hmul2(vl, *reinterpret_cast<const __half2*>(&s2bits));
        vh = __hmul2(vh, *reinterpret_cast<const __half2*>(&s2bits));
        out[16 * c + 4 * j + 2 * h] = *reinterpret_cast<uint32_t*>(&vl);
        out[16 * c + 4 * j + 2 * h + 1] = *reinterpret_cast<uint32_t*>(&vh);
      }
    }
  }
}

// int8: packed chunk c (16 bytes) holds K = 16c .. 16c+15 in byte order.  The
// per-row scale is applied to the fp32 accumulator in the epilogue, so the
// conversion is exact: (0x64 << 8 | (q + 128)) - 1152 in f16.
__device__ __forceinline__ void dequant_int8_row(const uint4 (&pk)[8], uint32_t (&out)[64]) {
  const uint32_t bias = 0x64806480u;  // 1152
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t w[4] = {pk[c].x, pk[c].y, pk[c].z, pk[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t u = w[j] ^ 0x80808080u;
      const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
      const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
      __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), *reinterpret_cast<const __half2*>(&bias));
      __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), *reinterpret_cast<const __half2*>(&bias));
      out[8 * c + 2 * j] = *reinterpret_cast<uint32_t*>(&a);
      out[8 * c + 2 * j + 1] = *reinterpret_cast<uint32_t*>(&b);
    }
  }
}

// The NK MMAs of one stage (K = 16 each) as one branch-free sequence: a branch
// between two tcgen05.mma instructions roughly triples their issue cost.  The
// A operand's K step kk is TMEM column a + 8kk; B's is 32 bytes along the
// 128-byte swizzled rows, with each 64-K block 1024 bytes after the previous.
template <int NK>
__device__ __forceinline__ void mma_stage(uint32_t d, uint32_t a, uint64_t bdesc0, uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int kk = 0; kk < NK; ++kk)
    mma_ts_f16(d, a + static_cast<uint32_t>(kk * 8), bdesc0 + static_cast<uint64_t>((kk >> 2) * 64 + (kk & 3) * 2),
               idesc, kk > 0 ? 1u : acc0);
}

__device__ __forceinline__ float silu_dev(float g) { return g / (1.0f + __expf(-g)); }

// Epilogue of 16 token columns [c0, c0+16) of one weight row (fp32 values with
// every scale applied).  Modes: SiLU(gate)*up into the fp32 intermediate
// (gate/up rows are adjacent lanes), fp32 gate/up partials, or the
// routing-weighted down output.
__device__ __forceinline__ void epilogue_store(const GemmParams& p, const WorkItem& it, int c0, int row, int lane,
                                               const float (&f)[16]) {
  if (p.epi_mode == kEpiSiluToAct) {
    // rows 2j / 2j+1 of the tile are gate / up of intermediate channel tile*64 + j
    const bool even = (lane & 1) == 0;
    const int jch = it.tile * (kTileRows / 2) + (row >> 1);
    float* inter = static_cast<float*>(p.out);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float send = even ? f[c + 8] : f[c];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
      const float gt = even ? f[c] : recv;
      const float up = even ? recv : f[c + 8];
      const int col = even ? c : c + 8;
      inter[static_cast<int64_t>(it.row0 + c0 + col) * p.inter_ld + jch] = silu_dev(gt) * up;
    }
  } else if (p.epi_mode == kEpiPartialRows) {
    float* h = static_cast<float*>(p.out) + it.split_idx * p.out_split_stride;
#pragma unroll
    for (int c = 0; c < 16; ++c) h[static_cast<int64_t>(it.row0 + c0 + c) * p.out_ld + it.tile * kTileRows + row] = f[c];
  } else {
    float* y = static_cast<float*>(p.out) + it.split_idx * p.out_split_stride;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int pair = __ldg(p.sorted_ids + it.row0 + c0 + c);
      if (pair < p.P)
        y[static_cast<int64_t>(pair) * p.out_ld + it.tile * kTileRows + row] = f[c] * __ldg(p.topk_w + pair);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.  TMEM columns: each of the two MMA issuers owns acc_bufs fp32
// accumulators of T columns (issuer i, buffer b at [(i*acc_bufs + b) * T]);
// the A stages (64*ks columns each) follow at a_col0.
// ---------------------------------------------------------------------------
template <bool INT4, bool BF16S>
__global__ void __launch_bounds__(kGemmThreads, 1) qmoe_gemm_kernel(const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int T = p.token_tile;
  const int KS = p.ks;
  const uint32_t b_bytes = static_cast<uint32_t>(T) * 256u * KS;
  const uint32_t st_bytes = gemm_stage_bytes(T, p.stage_bytes, KS);
  // NS and NA are even (the host plan guarantees it): stage g always lands in a
  // slot of parity g & 1, so each parity role sees every phase of its barriers.
  const int NS = p.smem_stages, NA = p.a_stages, ACCB = p.acc_bufs;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * st_bytes);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;
  uint64_t* aempty = afull + NA;
  uint64_t* accfull = aempty + NA;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;  // one per MMA issuer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 4 + 1);  // 4 dequant warps + 1 MMA commit
    }
    for (int j = 0; j < NA; ++j) {
      mbar_init(smem_u32(afull + j), 4);
      mbar_init(smem_u32(aempty + j), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(accfull + b), 2);   // one commit from each MMA issuer per item
      mbar_init(smem_u32(accempty + b), 4);  // the 4 epilogue warps
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(drain + 1), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // everything above overlaps the previous kernel; its results are read below
  pdl_launch_dependents();
  pdl_wait();

  const int nch = *p.n_chunks;
  const int n_items = nch * p.n_tiles * p.split;
  const uint32_t a_col0 = static_cast<uint32_t>(p.a_col0);

  if (warp == kProducerWarp || warp == kProducerWarp2) {
    // ------------------------------------------------------------ TMA producers
    // Two threads (warps 4 and 7) issue the copies of even and odd stages: issuing
    // one stage's copies takes one thread a few hundred cycles.
    if (lane == 0) {
      const int id = (warp == kProducerWarp) ? 0 : 1;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      Ring st;
      int g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        WorkItem it;
        decode_item(p, nch, i, it);
        const int64_t unit_w = static_cast<int64_t>(p.stage_bytes) * KS;
        const uint8_t* wsrc =
            p.w + (static_cast<int64_t>(it.e) * p.n_tiles + it.tile) * p.k_groups * static_cast<int64_t>(p.stage_bytes);
        // the chunk's rows of one stage of the pre-staged B operand: one contiguous run
        const uint32_t b_run = static_cast<uint32_t>(it.nrows) * 256u * KS;
        const uint8_t* bsrc = p.b + static_cast<int64_t>(it.row0) * 256 * KS;
        const uint32_t tx = static_cast<uint32_t>(unit_w) + b_run;
        for (int ks = it.ks0; ks < it.ks1; ++ks, ++g, st.next(NS)) {
          if ((g & 1) != id) continue;
          if (!mbar_wait(smem_u32(empty + st.idx), st.phase ^ 1u, abort_flag, 128)) {
            ok = false;
            break;
          }
          uint8_t* sp = smem + st.idx * st_bytes;
          const uint32_t fb = smem_u32(full + st.idx);
          mbar_arrive_expect_tx(fb, tx);
          if (!(p.fault_injection == 1 && blockIdx.x == 0 && g == 0)) {  // injected: armed, never filled
            tma_load_1d(smem_u32(sp + b_bytes), wsrc + ks * unit_w, static_cast<uint32_t>(unit_w), fb, pol_w);
            tma_load_1d(smem_u32(sp), bsrc + ks * p.b_unit_stride, b_run, fb, pol_b);
          }
        }
      }
      if (!ok) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
      // wait for every copy this thread may still have in flight into the CTA's shared memory
      // (its stages among the last NS before the first one it did not issue)
      for (int j = (g > NS ? g - NS : 0); j < g; ++j)
        if ((j & 1) == id) mbar_wait_drain(smem_u32(full + (j % NS)), (j / NS) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads (warps 5 and 6) issue the MMAs of even and odd stages into
    // their own accumulators: one thread's issue rate, with the waits and
    // commits around each stage, is below what the tensor core accepts at small
    // N, and the two run in parallel.
    if (lane == 0) {
      const int id = warp - kMmaWarp;
      Ring fr, ar;
      int g = 0, itn = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        WorkItem it;
        decode_item(p, nch, i, it);
        const uint32_t idesc = make_idesc_m128(static_cast<uint32_t>(it.nrows), false);
        const int b = (ACCB == 2) ? (itn & 1) : 0;
        const uint32_t use = (ACCB == 2) ? (itn >> 1) : itn;
        if (!mbar_wait(smem_u32(accempty + b), (use & 1u) ^ 1u, abort_flag, 16)) {
          ok = false;
          break;
        }
        const uint32_t d_tmem = tmem + static_cast<uint32_t>((id * ACCB + b) * T);
        uint32_t acc0 = 0u;  // the issuer's first stage of the item overwrites its accumulator
        for (int ks = it.ks0; ks < it.ks1; ++ks, ++g, fr.next(NS), ar.next(NA)) {
          if ((g & 1) != id) continue;
          if (!mbar_wait(smem_u32(full + fr.idx), fr.phase, abort_flag, 16) ||
              !mbar_wait(smem_u32(afull + ar.idx), ar.phase, abort_flag, 16)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem + a_col0 + static_cast<uint32_t>(ar.idx * 64 * KS);
          // B tile layout [8-row group][64-K block][8 rows][128 B]: 8-row groups are
          // 2048*ks bytes apart; later K steps only move the start address
          const uint64_t bdesc0 = make_sdesc_k_sw128(smem_u32(smem + fr.idx * st_bytes), 2048u * KS);
          if (KS == 2)
            mma_stage<16>(d_tmem, a_tmem, bdesc0, idesc, acc0);
          else
            mma_stage<8>(d_tmem, a_tmem, bdesc0, idesc, acc0);
          acc0 = 1u;
          mma_commit(smem_u32(empty + fr.idx));
          mma_commit(smem_u32(aempty + ar.idx));
        }
        if (!ok) break;
        // every issuer signals the item's end, also when it had no stage of it
        mma_commit(smem_u32(accfull + b));
        ++itn;
      }
      if (!ok) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
      // all MMAs this thread issued must finish before TMEM is released
      mma_commit(smem_u32(drain + id));
      mbar_wait_drain(smem_u32(drain + id), 0);
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant warpgroups
    const int wg = (warp - kDequantWarp0) >> 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    Ring fr, ar;
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      WorkItem it;
      decode_item(p, nch, i, it);
      for (int ks = it.ks0; ks < it.ks1; ++ks, ++g, fr.next(NS), ar.next(NA)) {
        if ((g & 1) != wg) continue;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(full + fr.idx), fr.phase, abort_flag));
        if (!ok) break;
        const uint8_t* wst = smem + fr.idx * st_bytes + b_bytes;
        const uint32_t ta = tmem + lane_base + a_col0 + static_cast<uint32_t>(ar.idx * 64 * KS);
        for (int j = 0; j < KS; ++j) {  // one 128-K group at a time: 64 TMEM columns each
          const uint8_t* wj = wst + j * p.stage_bytes;
          uint32_t out[64];
          if (INT4) {
            uint4 pk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) pk[c] = *reinterpret_cast<const uint4*>(wj + (c * 128 + row) * 16);
            const uint32_t sbits = *reinterpret_cast<const uint16_t*>(wj + 8192 + row * 2);
            if (j == KS - 1) {  // the stage's packed bytes are all in registers
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(empty + fr.idx));
            }
            dequant_int4_row<BF16S>(pk, sbits, out);
          } else {
            uint4 pk[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) pk[c] = *reinterpret_cast<const uint4*>(wj + (c * 128 + row) * 16);
            if (j == KS - 1) {
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(empty + fr.idx));
            }
            dequant_int8_row(pk, out);
          }
          if (j == 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(aempty + ar.idx), ar.phase ^ 1u, abort_flag));
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st_32x32b_x32<0>(ta + static_cast<uint32_t>(64 * j), out);
          tmem_st_32x32b_x32<32>(ta + static_cast<uint32_t>(64 * j + 32), out);
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(afull + ar.idx));
      }
    }
    if (!ok && lane == 0) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue warpgroup
    const int q = warp;
    const int row = q * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int itn = 0, g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      WorkItem it;
      decode_item(p, nch, i, it);
      const int b = (ACCB == 2) ? (itn & 1) : 0;
      const uint32_t use = (ACCB == 2) ? (itn >> 1) : itn;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(accfull + b), use & 1u, abort_flag, 512));
      if (!ok) break;
      tc_fence_after();
      // issuer 0 took the item's even global stages, issuer 1 the odd ones
      const int n_st = it.ks1 - it.ks0;
      const bool has0 = n_st >= 2 || (g & 1) == 0;
      const bool has1 = n_st >= 2 || (g & 1) == 1;
      g += n_st;
      const float rs =
          INT4 ? 1.0f : __ldg(p.row_scale + (static_cast<int64_t>(it.e) * p.n_tiles + it.tile) * kTileRows + row);
      const uint32_t t0 = tmem + lane_base + static_cast<uint32_t>(b * T);
      const uint32_t t1 = tmem + lane_base + static_cast<uint32_t>((ACCB + b) * T);
      for (int c0 = 0; c0 < it.nrows; c0 += 16) {
        uint32_t v[16], w[16];
        if (has0) tmem_ld_32x32b_x16(t0 + static_cast<uint32_t>(c0), v);
        if (has1) tmem_ld_32x32b_x16(t1 + static_cast<uint32_t>(c0), w);
        tmem_wait_ld();
        if (c0 + 16 >= it.nrows) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(accempty + b));
        }
        float f[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float cs = __ldg(p.col_scale + it.row0 + c0 + c);
          f[c] = ((has0 ? __uint_as_float(v[c]) : 0.0f) + (has1 ? __uint_as_float(w[c]) : 0.0f)) * rs * cs;
        }
        epilogue_store(p, it, c0, row, lane, f);
      }
      ++itn;
    }
    if (!ok && lane == 0) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool INT4, bool BF16S>
cudaError_t launch_gemm_t(const GemmParams& p, int grid, cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(p);
  cudaError_t err = cudaFuncSetAttribute(qmoe_gemm_kernel<INT4, BF16S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_kernel(qmoe_gemm_kernel<INT4, BF16S>, dim3(grid), dim3(kGemmThreads), smem, stream, true, p);
}

}  // namespace qmoe
