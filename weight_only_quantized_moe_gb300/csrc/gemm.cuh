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
//   * one pipeline stage = one 128-K quantization group.  Three rings: packed
//     weights in shared memory (deep: they stream from HBM), token tiles in
//     shared memory (token tiles come from L2) and dequantized A tiles in
//     TMEM.  The token-tile ring is a multiple (1 to 3) of the A ring, so a
//     token tile is fetched several stages before its MMAs and its L2 latency
//     stays off the A slots' cycle.  Weights and token tiles arrive by 1-D
//     bulk TMA copies: the producers of the B operand (gather, rescale) store
//     it pre-staged, per 128-K group and 8-row group, in the 128-byte-swizzled
//     K-major layout the MMA's shared-memory descriptor reads, so a chunk's
//     tile for one stage is one contiguous run.
//   * warp roles (25 warps): two TMA producer threads (warps 4, 7) take the
//     even and the odd stages; the dequant warps 8-23 form four sets of four
//     (stage g to set g mod 4; each warp converts whole stage rows for the 32
//     rows of its TMEM lane quadrant) or two sets of eight (half rows).  The
//     MMAs are issued by warps 5 and 6 (stage g to issuer g mod NI, each with
//     its own accumulator; warp 24 is a third issuer on request), each warp
//     converged with one elected lane issuing, while the token tile is small
//     and one warp's issue rate is the limit, and by warp 5 alone when the
//     tile is large and the tensor pipe is, so that two accumulator buffers
//     fit in TMEM.  Warps 0-3 are the epilogue.  A persistent grid walks the
//     work items.
//   * CTA pairs (PAIR): clusters of two CTAs on two SMs walk the same items,
//     each with a pair of 128-row weight tiles; each CTA dequantizes its own
//     tile into its own TMEM and copies half of the token tile's rows, and the
//     even CTA issues M = 256 MMAs (cta_group::2) over both, with commits
//     multicast to both CTAs; the odd CTA's dequant sets and epilogue warps
//     arrive on the even CTA's A and accumulator barriers.
//   * barriers per stage: the dequant set waits for the weights and the token
//     tile (one barrier counts both copies), releases the weight slot,
//     converts, waits until the MMAs of the stage that last used its A slot
//     are done (implied by the token tile's arrival when both rings have the
//     same depth), writes A and signals it; the issuer waits for that one
//     signal, issues the stage's MMAs and commits one "stage done" barrier,
//     which frees the stage's A slot and its token-tile slot.  Every ring's
//     size is a multiple of the stride of each role that uses it (2 for
//     producers and dequant sets, NI for the issuers), so each slot belongs
//     to one role of each kind and each role sees every phase of the barriers
//     it waits on.
//   * every mbarrier wait is bounded (see ptx.cuh); a wait that gives up
//     records QMOE_ERR_TIMEOUT in the status word and the CTA winds down after
//     waiting for its own copies and MMAs, then frees its TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qmoe_internal.h"

namespace qmoe {

constexpr int kGemmThreads = 800;  // 25 warps
constexpr int kProducerWarp = 4;
constexpr int kProducerWarp2 = 7;
constexpr int kMmaWarp = 5;        // issuers 0 and 1: warps 5 and 6; issuer 2: warp 24
constexpr int kMmaWarp3 = 24;
constexpr int kDequantWarp0 = 8;   // warps 8..23: two sets of 8 or four sets of 4
constexpr int kMaxIssuers = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescSparse = 1u << 2;  // instruction descriptor: A is 2:4 structured sparse
constexpr int kBarrierBytes = 1024;

__host__ __device__ inline uint32_t gemm_w_slot(int group_bytes) { return (group_bytes + 1023u) & ~1023u; }
// Bytes of one token-tile ring slot: the tile's rows of one 128-K stage (a CTA of
// a pair holds half of them).
__host__ __device__ inline uint32_t gemm_b_slot(int token_tile, bool pair) {
  return static_cast<uint32_t>(token_tile) * (pair ? 128u : 256u);
}
// Dynamic shared memory: weight ring, token-tile ring, barriers, the per-group
// staging buffers (per-group-scaled int4 only), +1 KB alignment slack.
__host__ __device__ inline size_t gemm_smem_layout_bytes(int w_stages, int group_bytes, int b_stages, int token_tile,
                                                         bool pg, bool pair) {
  return 1024 + static_cast<size_t>(w_stages) * gemm_w_slot(group_bytes) +
         static_cast<size_t>(b_stages) * gemm_b_slot(token_tile, pair) + kBarrierBytes + (pg ? kPgStageBytes : 0);
}

struct WorkItem {
  int e, row0, nrows, tile, split_idx, ks0, ks1;
  bool phantom;  // CTA pair, odd tile count: the odd CTA's tile of the last pair does not exist
};

// Work item i -> (split, chunk, tile).  Items of one split are rastered in
// groups of chunks with the tile varying slowest inside a group, so that the
// CTAs running at the same time share the group's token tiles and each weight
// tile in L2.  chunk_group > 0: groups of that many consecutive chunks (decode:
// one chunk per expert, several experts per group).  chunk_group = -G: every
// group is a piece of at most G chunks of one expert (large batches: each
// weight tile is then read once per piece, while the piece's token tiles stay
// in L2); group (start s, n chunks) owns items [s, s + n) x n_tiles, so the
// chunk at item / n_tiles names the group.  On CTA pairs the items run over tile
// pairs instead of tiles, and CTA `rank` of the pair takes tile 2 * pair + rank;
// with an odd tile count the last pair's odd tile is a phantom: that CTA reads
// the last real tile again (the pair MMA needs its A rows and its half of the
// token rows) and stores nothing.
template <bool PAIR>
__device__ __forceinline__ void decode_item(const GemmParams& p, int nch, int i, uint32_t rank, WorkItem& w) {
  const int n_units = PAIR ? (p.n_tiles + 1) >> 1 : p.n_tiles;
  const int per_split = nch * n_units;
  const int s = i / per_split;
  const int r = i - s * per_split;
  int c0, cg;
  if (p.chunk_group > 0) {
    const int grp_items = p.chunk_group * n_units;
    c0 = (r / grp_items) * p.chunk_group;
    cg = min(p.chunk_group, nch - c0);
  } else {
    const int G = -p.chunk_group;
    const Chunk cu = p.chunks[r / n_units];
    const int piece = (r / n_units - cu.first) / G;
    c0 = cu.first + piece * G;
    cg = min(G, cu.count - piece * G);
  }
  const int rem = r - c0 * n_units;
  const int unit = rem / cg;
  const int c = c0 + (rem - unit * cg);
  const Chunk ch = p.chunks[c];
  const int tile = PAIR ? 2 * unit + static_cast<int>(rank) : unit;
  w.e = ch.expert;
  w.row0 = ch.row0;
  w.nrows = ch.nrows;
  w.phantom = PAIR && tile >= p.n_tiles;
  w.tile = w.phantom ? p.n_tiles - 1 : tile;
  w.split_idx = s;
  w.ks0 = static_cast<int>(static_cast<int64_t>(p.k_groups) * s / p.split);
  w.ks1 = static_cast<int>(static_cast<int64_t>(p.k_groups) * (s + 1) / p.split);
}

// First stage index >= g0 that a role taking every r-th stage from stage `phase` owns.
__device__ __forceinline__ int first_own(int g0, int phase, int r) {
  int m = (phase - g0) % r;
  if (m < 0) m += r;
  return g0 + m;
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
// Dequantization of half a stage row (64 K) into 32 TMEM columns (column c
// holds K elements 2c (low half) and 2c+1 (high half)), as f16.
// ---------------------------------------------------------------------------
// int4: packed chunk c (16 bytes) of the row holds K = 32c .. 32c+31; in word j
// of the chunk, nibble i holds K = 32c+8j+2i and nibble i+4 holds K = 32c+8j+2i+1.
// Magic-number conversion: (nibble | 0x6400) is the f16 value 1024 + q, exact,
// and subtracting 1032 gives q - 8 exactly; nibbles i = 1, 3 stay in bits 4..7
// of their half, where (nibble << 4) | 0x6400 is 1024 + 16q and
// fma(v, 1/16, -72) = q - 8 exactly, so one shift per word serves i = 2, 3.
// One multiply by the group scale rounds once (exact for bf16 scales).
// `pk` holds chunks 2h and 2h+1 of the row for half h.  With a zero point z
// (0..15; 8 for the symmetric format) the two constants become 1024 + z and
// -(64 + z), still exact, so zero points cost no instruction.
// One 32-bit word's two nibble pairs (lo: bits 0..3 / 16..19, hi: bits 4..7 /
// 20..23 of `src`) to two f16x2 values (q - z) * s: two LOP3, one subtract, one
// FMA and two multiplies, written out so that nothing else is generated.
__device__ __forceinline__ void cvt_int4_word_half(uint32_t src, uint32_t bias, uint32_t m64z, uint32_t s2,
                                                   uint32_t& lo_out, uint32_t& hi_out) {
  asm("{\n\t.reg .b32 lo, hi;\n\t"
      "lop3.b32 lo, %2, 0x000F000F, 0x64006400, 0xEA;\n\t"   // (src & mask) | 0x6400: 1024 + q
      "lop3.b32 hi, %2, 0x00F000F0, 0x64006400, 0xEA;\n\t"   // 1024 + 16 q
      "sub.rn.f16x2 lo, lo, %3;\n\t"                        // q - z
      "fma.rn.f16x2 hi, hi, %6, %4;\n\t"                    // (1024 + 16q) / 16 - (64 + z) = q - z
      "mul.rn.f16x2 %0, lo, %5;\n\t"
      "mul.rn.f16x2 %1, hi, %5;\n\t}"
      : "=r"(lo_out), "=r"(hi_out)
      : "r"(src), "r"(bias), "r"(m64z), "r"(s2), "r"(0x2C002C00u));
}

// One 16-byte chunk of a row (32 K) to 16 f16x2 values (q - z) * s.  Constants:
// bias_bits = 1024 + z and m64z = -(64 + z) as f16x2 (see int4_zp_constants),
// s2bits = the f16 scale in both halves (int4_scale_pair).
__device__ __forceinline__ void dequant_int4_chunk(const uint4& pk, uint32_t bias_bits, uint32_t m64z, uint32_t s2bits,
                                                   uint32_t (&out)[16]) {
  const uint32_t w[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cvt_int4_word_half(w[j], bias_bits, m64z, s2bits, out[4 * j], out[4 * j + 1]);
    cvt_int4_word_half(w[j] >> 8, bias_bits, m64z, s2bits, out[4 * j + 2], out[4 * j + 3]);
  }
}

__device__ __forceinline__ void int4_zp_constants(uint32_t z, uint32_t& bias_bits, uint32_t& m64z) {
  bias_bits = 0x64006400u | z | (z << 16);  // 1024 + z
  m64z = 0xD400D400u | (z << 4) | (z << 20);  // -(64 + z)
}

// The group scale as an f16 pair (a bf16 scale is rounded to f16 once).
template <bool BF16S>
__device__ __forceinline__ uint32_t int4_scale_pair(uint32_t sbits) {
  const uint16_t s16 = BF16S ? __half_as_ushort(__float2half_rn(__uint_as_float(sbits << 16)))
                             : static_cast<uint16_t>(sbits);
  return static_cast<uint32_t>(s16) | (static_cast<uint32_t>(s16) << 16);
}

// int8: packed chunk c (16 bytes) holds K = 16c .. 16c+15 in byte order.  The
// conversion is exact: (0x64 << 8 | (q + 128)) - 1152 in f16.  A per-row
// (per-column of W) scale is applied to the fp32 accumulator in the epilogue;
// a group scale (GS) multiplies here, rounding once.  `pk` holds chunks
// 4h .. 4h+3 of the row for half h.
// One 32-bit word (4 int8 codes) to two f16x2 values: flip the sign bit
// (q + 128), place each byte under the exponent 0x64 (1024 + q + 128) and
// subtract 1152; with a group scale, multiply.
template <bool GS>
__device__ __forceinline__ void cvt_int8_word(uint32_t w, uint32_t s2, uint32_t& a_out, uint32_t& b_out) {
  if (GS) {
    asm("{\n\t.reg .b32 u, lo, hi;\n\t"
        "xor.b32 u, %2, 0x80808080;\n\t"
        "prmt.b32 lo, u, 0x64646464, 0x4140;\n\t"
        "prmt.b32 hi, u, 0x64646464, 0x4342;\n\t"
        "sub.rn.f16x2 lo, lo, %3;\n\t"
        "sub.rn.f16x2 hi, hi, %3;\n\t"
        "mul.rn.f16x2 %0, lo, %4;\n\t"
        "mul.rn.f16x2 %1, hi, %4;\n\t}"
        : "=r"(a_out), "=r"(b_out)
        : "r"(w), "r"(0x64806480u), "r"(s2));
  } else {
    asm("{\n\t.reg .b32 u, lo, hi;\n\t"
        "xor.b32 u, %2, 0x80808080;\n\t"
        "prmt.b32 lo, u, 0x64646464, 0x4140;\n\t"
        "prmt.b32 hi, u, 0x64646464, 0x4342;\n\t"
        "sub.rn.f16x2 %0, lo, %3;\n\t"
        "sub.rn.f16x2 %1, hi, %3;\n\t}"
        : "=r"(a_out), "=r"(b_out)
        : "r"(w), "r"(0x64806480u));
  }
}

template <bool GS, bool BF16S>
__device__ __forceinline__ void dequant_int8_half(const uint4 (&pk)[4], uint32_t sbits, uint32_t (&out)[32]) {
  uint32_t s2bits = 0;
  if (GS) {
    const uint16_t s16 =
        BF16S ? __half_as_ushort(__float2half_rn(__uint_as_float(sbits << 16))) : static_cast<uint16_t>(sbits);
    s2bits = static_cast<uint32_t>(s16) | (static_cast<uint32_t>(s16) << 16);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {pk[c].x, pk[c].y, pk[c].z, pk[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) cvt_int8_word<GS>(w[j], s2bits, out[8 * c + 2 * j], out[8 * c + 2 * j + 1]);
  }
}

// Per-group-scaled int4 (16-row token tiles, zero point 8): half a stage row to
// 32 TMEM columns of raw magic-number halves, 1024 + q at the low nibble of each
// byte pair and 1024 + 16 q at the high one (two LOP3 per word and one shift for
// the second pair); the scale, the zero point and the 1/16 are applied later, per
// stage, by the epilogue (see the gather's per-group corrections).
__device__ __forceinline__ void dequant_int4_raw_half(const uint4 (&pk)[2], uint32_t (&out)[32]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t w[4] = {pk[c].x, pk[c].y, pk[c].z, pk[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w8 = w[j] >> 8;
      asm("lop3.b32 %0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
          "lop3.b32 %1, %4, 0x00F000F0, 0x64006400, 0xEA;\n\t"
          "lop3.b32 %2, %5, 0x000F000F, 0x64006400, 0xEA;\n\t"
          "lop3.b32 %3, %5, 0x00F000F0, 0x64006400, 0xEA;"
          : "=r"(out[16 * c + 4 * j]), "=r"(out[16 * c + 4 * j + 1]), "=r"(out[16 * c + 4 * j + 2]),
            "=r"(out[16 * c + 4 * j + 3])
          : "r"(w[j]), "r"(w8));
    }
  }
}

// 2:4-sparse formats: a row's half (64 K, 16 groups of 4 channels) holds the two
// kept codes of each group and their positions.  The kept codes become 16 f16x2
// values, value g = (first, second) kept value of group g, and go to tensor memory
// as the structured-sparse MMA's A operand; the MMA reads the positions from the
// metadata words the packer stores in its lane order, so no placement work is
// done here.  int4: word j of the 16 code bytes holds groups 4j..4j+3 with nibble i
// the first kept code of group 4j+i and nibble i+4 its second, so the int4
// conversion turns each word into the values of four groups.  int8: word j of the
// 32 code bytes holds groups 2j and 2j+1 as bytes (first, second) of each.
template <bool BF16S>
__device__ __forceinline__ void dequant_int4_24_vals_half(const uint4& pk, uint32_t sbits, uint32_t (&out)[16]) {
  const uint32_t bias_bits = 0x64086408u;  // 1024 + 8
  const uint32_t m64z = 0xD480D480u;       // -(64 + 8)
  const uint16_t s16 = BF16S ? __half_as_ushort(__float2half_rn(__uint_as_float(sbits << 16))) : static_cast<uint16_t>(sbits);
  const uint32_t s2bits = static_cast<uint32_t>(s16) | (static_cast<uint32_t>(s16) << 16);
  const uint32_t w[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    cvt_int4_word_half(w[j], bias_bits, m64z, s2bits, out[4 * j], out[4 * j + 1]);
    cvt_int4_word_half(w[j] >> 8, bias_bits, m64z, s2bits, out[4 * j + 2], out[4 * j + 3]);
  }
}

template <bool GS, bool BF16S>
__device__ __forceinline__ void dequant_int8_24_vals_half(const uint4 (&pk)[2], uint32_t sbits, uint32_t (&out)[16]) {
  uint32_t s2bits = 0;
  if (GS) {
    const uint16_t s16 =
        BF16S ? __half_as_ushort(__float2half_rn(__uint_as_float(sbits << 16))) : static_cast<uint16_t>(sbits);
    s2bits = static_cast<uint32_t>(s16) | (static_cast<uint32_t>(s16) << 16);
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint32_t w[4] = {pk[c].x, pk[c].y, pk[c].z, pk[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) cvt_int8_word<GS>(w[j], s2bits, out[8 * c + 2 * j], out[8 * c + 2 * j + 1]);
  }
}

// The 4 sparse MMAs of one stage (K = 32 of the dense matrix each): the A slot holds
// the kept values in columns 0..31 (8 per MMA) and MMA kk's position words in
// column 32 + 8 kk (8-column aligned, as the A operand's steps).
__device__ __forceinline__ void mma_stage_sp(uint32_t issue, uint32_t d, uint32_t a, uint64_t bdesc0, uint32_t idesc,
                                             uint32_t acc0) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts_sp_f16(issue, d, a + static_cast<uint32_t>(kk * 8), bdesc0 + static_cast<uint64_t>((kk >> 1) * 64 + (kk & 1) * 4),
                  a + 32u + static_cast<uint32_t>(8 * kk), idesc, kk > 0 ? 1u : acc0);
}

// The 8 MMAs of one stage (K = 16 each) as one branch-free sequence: a branch
// between two tcgen05.mma instructions roughly triples their issue cost.  The
// A operand's K step kk is TMEM column a + 8kk; B's is 32 bytes along the
// 128-byte swizzled rows, the second 64-K block 1024 bytes after the first.
// Executed by the whole issuer warp; the lane with `issue` set issues (M = 256
// pair MMAs from a CTA pair's even CTA).
template <bool PAIR>
__device__ __forceinline__ void mma_stage(uint32_t issue, uint32_t d, uint32_t a, uint64_t bdesc0, uint32_t idesc,
                                          uint32_t acc0) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ak = a + static_cast<uint32_t>(kk * 8);
    const uint64_t bk = bdesc0 + static_cast<uint64_t>((kk >> 2) * 64 + (kk & 3) * 2);
    if constexpr (PAIR)
      mma_ts_f16_pair(issue, d, ak, bk, idesc, kk > 0 ? 1u : acc0);
    else
      mma_ts_f16(issue, d, ak, bk, idesc, kk > 0 ? 1u : acc0);
  }
}

__device__ __forceinline__ float silu_dev(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Top-k reduction in the down GEMM's epilogue.  Output element (token m, feature
// n) is the sum over m's valid experts j and the K splits s of the partials
// y[s][m*top_k + j][n], which several items (CTAs) write.  Each epilogue warp,
// after storing its 32 rows of 16 token columns, counts one arrival per column
// on the (token, 128-row tile, lane quadrant) counter; the warp whose arrival
// completes the count (valid experts x splits) sums that token's 32 rows in the
// fixed order (j, then s) of the separate reduce kernel and writes them.  No
// warp waits for another: the fences order every partial store before its
// arrival and the final reads after the last one.
static __device__ __noinline__ void reduce_topk(const GemmParams& p, const WorkItem& it, int c0, int row, int lane) {
  __threadfence();
  __syncwarp();
  int m = -1;
  bool last = false;
  if (lane < 16) {
    const int pair = __ldg(p.sorted_ids + it.row0 + c0 + lane);
    if (pair < p.P) {
      m = pair / p.top_k;
      int need = 0;
      for (int j = 0; j < p.top_k; ++j) {
        const int e = __ldg(p.topk_ids + static_cast<int64_t>(m) * p.top_k + j);
        need += (e >= 0 && e < p.n_experts) ? 1 : 0;
      }
      need *= p.split;
      const int64_t ci = (static_cast<int64_t>(m) * p.n_tiles + it.tile) * 4 + (row >> 5);
      last = atomicAdd(p.red_cnt + ci, 1) == need - 1;
    }
  }
  unsigned todo = __ballot_sync(0xffffffffu, last);
  if (todo == 0) return;
  __threadfence();
  const int64_t n = static_cast<int64_t>(it.tile) * kTileRows + row;
  const float* y0 = static_cast<const float*>(p.out);
  while (todo != 0) {
    const int c = __ffs(todo) - 1;
    todo &= todo - 1;
    const int mm = __shfl_sync(0xffffffffu, m, c);
    float acc = 0.0f;
    for (int j = 0; j < p.top_k; ++j) {
      const int e = __ldg(p.topk_ids + static_cast<int64_t>(mm) * p.top_k + j);
      if (e < 0 || e >= p.n_experts) continue;
      const float* yp = y0 + (static_cast<int64_t>(mm) * p.top_k + j) * p.out_ld + n;
      for (int s = 0; s < p.split; ++s) acc += __ldcg(yp + s * p.out_split_stride);
    }
    p.red_out[static_cast<int64_t>(mm) * p.out_ld + n] =
        p.out_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(acc)) : __half_as_ushort(__float2half_rn(acc));
  }
}

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
  } else if (p.epi_mode == kEpiLinearOut) {
    // dense linear: B row r is token r (rows >= P are padding); out[r, n] in the activation type
    uint16_t* o = static_cast<uint16_t*>(p.out);
    const int n = it.tile * kTileRows + row;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int r = it.row0 + c0 + c;
      if (r < p.P) {
        const uint16_t v = p.out_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f[c]))
                                      : __half_as_ushort(__float2half_rn(f[c]));
        o[static_cast<int64_t>(r) * p.out_ld + n] = v;
      }
    }
  } else {
    float* y = static_cast<float*>(p.out) + it.split_idx * p.out_split_stride;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int pair = __ldg(p.sorted_ids + it.row0 + c0 + c);
      if (pair < p.P)
        y[static_cast<int64_t>(pair) * p.out_ld + it.tile * kTileRows + row] = f[c] * __ldg(p.topk_w + pair);
    }
    if (p.red_cnt != nullptr) reduce_topk(p, it, c0, row, lane);
  }
}

// ---------------------------------------------------------------------------
// The kernel.  Shared memory: weight ring (w_stages slots), token-tile ring
// (b_stages slots of T rows), barriers.  TMEM columns: issuer i owns acc_bufs
// fp32 accumulators of T columns at [(i*acc_bufs + b) * T]; stage g uses the
// 64-column A slot a_col0 + 64 (g mod ab_stages) and the token-tile slot
// g mod b_stages, whose "done" barrier the issuer commits.  Every role walks
// only its own stages (every 2nd for producers and dequant sets, every NI-th
// for the MMA issuers), stepping its ring positions by the same stride.
// ---------------------------------------------------------------------------
template <int KIND, bool BF16S, bool PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1) qmoe_gemm_kernel(const GemmParams p) {
  constexpr bool INT4 = KIND == kQ4 || KIND == kQ4Z || KIND == kQ4P;
  constexpr bool PG = KIND == kQ4P;  // per-group scaling in the epilogue
  constexpr bool SPARSE = KIND == kQ4S || KIND == kQ8S || KIND == kQ8SG;
  static_assert(!PAIR || (!PG && !SPARSE), "CTA pairs run the dense formats with the standard epilogue");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int T = p.token_tile;
  const int NW = p.w_stages, NB = p.ab_stages, NB2 = p.b_stages, ACCB = p.acc_bufs, NI = p.issuers;
  const uint32_t wslot = gemm_w_slot(p.stage_bytes);
  const uint32_t bslot = gemm_b_slot(T, PAIR);
  uint8_t* wring = smem;
  uint8_t* bring = smem + NW * wslot;

  // wfull[i] completes when a stage's weights AND its token tile have landed (the
  // producer arms it for both copies; the token-tile copy, issued later, counts on it)
  uint64_t* wfull = reinterpret_cast<uint64_t*>(bring + NB2 * bslot);
  uint64_t* wempty = wfull + NW;
  uint64_t* afull = wempty + NW;
  // done[j]: the MMAs of the stage in token-tile slot j completed, so that
  // slot and the stage's A slot are free again
  uint64_t* done = afull + NB;
  uint64_t* accfull = done + NB2;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;  // one per MMA issuer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + kMaxIssuers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: both CTAs of a cluster walk the same items and stages; rank 0
  // issues the pair's MMAs
  const uint32_t rank = PAIR ? cluster_cta_rank() : 0u;
  const int item0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int item_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    const uint32_t wps = 16u / static_cast<uint32_t>(p.dq_sets);  // warps of a dequant set
    for (int s = 0; s < NW; ++s) {
      mbar_init(smem_u32(wfull + s), 1);
      mbar_init(smem_u32(wempty + s), wps);
    }
    // with per-group scaling the 4 epilogue warps also release each A slot's D slot;
    // on CTA pairs the even CTA's A and accumulator barriers count both CTAs' warps
    for (int j = 0; j < NB; ++j) mbar_init(smem_u32(afull + j), (PAIR ? 2u : 1u) * wps + (PG ? 4u : 0u));
    for (int j = 0; j < NB2; ++j) mbar_init(smem_u32(done + j), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(accfull + b), NI);               // one commit from each MMA issuer per item
      mbar_init(smem_u32(accempty + b), PAIR ? 8u : 4u);  // the 4 epilogue warps (of each CTA)
    }
    for (int i = 0; i < kMaxIssuers; ++i) mbar_init(smem_u32(drain + i), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrive
  if (warp == kMmaWarp) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // everything above overlaps the previous kernel; its results are read below
  pdl_launch_dependents();
  pdl_wait();

  const int nch = *p.n_chunks;
  const int n_items = nch * (PAIR ? (p.n_tiles + 1) >> 1 : p.n_tiles) * p.split;
  const uint32_t a_col0 = static_cast<uint32_t>(p.a_col0);

  if (warp == kProducerWarp || warp == kProducerWarp2) {
    // ------------------------------------------------------------ TMA producers
    // Two threads (warps 4 and 7) issue the copies of even and odd stages.
    if (lane == 0) {
      const int id = (warp == kProducerWarp) ? 0 : 1;
      // weights read by one CTA stream through L2 (evict first); weights shared by
      // several chunks of one expert stay for the co-scheduled CTAs (evict normal)
      const uint64_t pol_w = p.w_shared ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      Ring wr, br;
      wr.idx = br.idx = id;
      int g0 = 0, last_w = -1, last_b = -1;
      bool ok = true;
      for (int i = item0; i < n_items && ok; i += item_step) {
        WorkItem it;
        decode_item<PAIR>(p, nch, i, rank, it);
        const int n_st = it.ks1 - it.ks0;
        const uint8_t* wsrc =
            p.w + (static_cast<int64_t>(it.e) * p.n_tiles + it.tile) * p.k_groups * static_cast<int64_t>(p.stage_bytes);
        // the chunk's rows of one stage of the pre-staged B operand: one contiguous run
        // (a CTA pair's CTA: its half of the rows, whole 8-row groups as chunks hold
        // multiples of 16 rows)
        const uint32_t b_run = static_cast<uint32_t>(it.nrows) * (PAIR ? 128u : 256u);
        const uint8_t* bsrc =
            p.b + (static_cast<int64_t>(it.row0) + static_cast<int64_t>(rank) * (it.nrows >> 1)) * 256;
        for (int g = first_own(g0, id, 2); g < g0 + n_st; g += 2, wr.step(2, NW), br.step(2, NB2)) {
          const int ks = it.ks0 + (g - g0);
          const bool inject = p.fault_injection == 1 && blockIdx.x == 0 && g == 0;  // armed, never filled
          if (!mbar_wait(smem_u32(wempty + wr.idx), wr.phase ^ 1u, abort_flag, 128)) {
            ok = false;
            break;
          }
          const uint32_t wb = smem_u32(wfull + wr.idx);
          mbar_arrive_expect_tx(wb, static_cast<uint32_t>(p.stage_bytes) + b_run);
          if (!inject)
            tma_load_1d(smem_u32(wring + wr.idx * wslot), wsrc + static_cast<int64_t>(ks) * p.stage_bytes,
                        static_cast<uint32_t>(p.stage_bytes), wb, pol_w);
          last_w = g;
          // the token-tile slot is free once the MMAs of its previous stage completed
          if (!mbar_wait(smem_u32(done + br.idx), br.phase ^ 1u, abort_flag, 128)) {
            ok = false;
            break;
          }
          if (!inject) tma_load_1d(smem_u32(bring + br.idx * bslot), bsrc + ks * p.b_unit_stride, b_run, wb, pol_b);
          last_b = g;
        }
        g0 += n_st;
      }
      if (!ok) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
      // wait for every copy this thread may still have in flight into the CTA's shared
      // memory: both copies of a stage count on its wfull barrier, so the stages
      // among the last NW it armed cover them (a stage whose token-tile copy was
      // never issued after an abort leaves its barrier pending: the drain wait
      // then runs into its time limit, with no copy in flight)
      (void)last_b;
      for (int j = (last_w >= NW ? last_w - NW + 2 : id); j <= last_w; j += 2)
        mbar_wait_drain(smem_u32(wfull + (j % NW)), (j / NW) & 1);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1 || warp == kMmaWarp3) {
    // ------------------------------------------------------------ MMA issuers
    // With NI issuers, issuer i takes stages i, i+NI, ... into its own
    // accumulator: one warp's MMA issue rate, with the wait and commit around
    // each stage, is below what the tensor core accepts at small N.  With one
    // (large tiles) warp 5 takes every stage.
    const int id = (warp == kMmaWarp3) ? 2 : warp - kMmaWarp;
    // The whole warp walks the loop, converged, and one elected lane issues: the
    // slot addresses and descriptors then stay warp-uniform.
    // On CTA pairs the even CTA issues M = 256 MMAs for both and multicasts its
    // commits to both CTAs' barriers.
    auto commit = [&](uint32_t issue, uint32_t bar) {
      if constexpr (PAIR)
        mma_commit_pair(issue, bar);
      else
        mma_commit(issue, bar);
    };
    if (id < NI && rank == 0) {
      const uint32_t issue = elect_one_sync();
      Ring ar, br;  // A slot (NB) and token-tile slot / done barrier (NB2) of the stage
      ar.idx = br.idx = id;
      int g0 = 0, itn = 0;
      bool ok = true;
      for (int i = item0; i < n_items && ok; i += item_step) {
        WorkItem it;
        decode_item<PAIR>(p, nch, i, rank, it);
        const int n_st = it.ks1 - it.ks0;
        const uint32_t idesc = PAIR ? make_idesc_m256(static_cast<uint32_t>(it.nrows), false)
                                    : make_idesc_m128(static_cast<uint32_t>(it.nrows), false);
        const int b = (ACCB == 2) ? (itn & 1) : 0;
        const uint32_t use = (ACCB == 2) ? (itn >> 1) : itn;
        if (!PG) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(accempty + b), (use & 1u) ^ 1u, abort_flag, 16));
          if (!ok) break;
        }
        const uint32_t d_acc = tmem + static_cast<uint32_t>((id * ACCB + b) * T);
        uint32_t acc0 = 0u;  // the issuer's first stage of the item overwrites its accumulator
        for (int g = first_own(g0, id, NI); g < g0 + n_st; g += NI, ar.step(NI, NB), br.step(NI, NB2)) {
          // the dequant set signals A only after the stage's token tile has landed
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(afull + ar.idx), ar.phase, abort_flag, 16));
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_tmem = tmem + a_col0 + static_cast<uint32_t>(ar.idx * 64);
          // token tile [8-row group][64-K block][8 rows][128 B]: 8-row groups 2048 bytes apart
          const uint64_t bdesc0 = make_sdesc_k_sw128(smem_u32(bring + br.idx * bslot), 2048u);
          if (SPARSE) {
            mma_stage_sp(issue, d_acc, a_tmem, bdesc0, idesc | kIdescSparse, acc0);
          } else if (PG) {
            // per-group scaling: the stage's sum goes to the D slot of its A slot, fresh
            mma_stage<PAIR>(issue, tmem + static_cast<uint32_t>(p.d_col0) + static_cast<uint32_t>(ar.idx * 16),
                            a_tmem, bdesc0, idesc, 0u);
          } else {
            mma_stage<PAIR>(issue, d_acc, a_tmem, bdesc0, idesc, acc0);
          }
          acc0 = 1u;
          commit(issue, smem_u32(done + br.idx));
        }
        if (!ok) break;
        // every issuer signals the item's end, also when it had no stage of it
        if (!PG) commit(issue, smem_u32(accfull + b));
        g0 += n_st;
        ++itn;
      }
      if (!ok && issue) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
      // all MMAs this warp issued must finish before TMEM is released (in both CTAs of a pair)
      commit(issue, smem_u32(drain + id));
      mbar_wait_drain(smem_u32(drain + id), 0);
    } else if (PAIR && id < NI) {
      // a pair's odd CTA: its TMEM and shared memory stay in use until the even
      // CTA's issuer reports all its MMAs complete
      mbar_wait_drain(smem_u32(drain + id), 0);
    }
  } else if (warp >= kDequantWarp0) {
    // ------------------------------------------------------------ dequant sets
    // DS sets of 16/DS warps; set s takes stages s, s + DS, ...  With 2 sets a
    // warp converts one K half of its 32 rows (its TMEM lane quadrant); with 4
    // sets a warp converts both halves of its rows, which halves the per-stage
    // wait / store / arrive work and keeps four stages in conversion at once.
    const int DS = p.dq_sets;
    const int wps = 16 / DS;
    const int dw = warp - kDequantWarp0;
    const int set = dw / wps;
    const int q = warp & 3;                                  // TMEM lane quadrant = rows 32q .. 32q+31
    const int h0 = (wps == 8) ? ((dw >> 2) & 1) : 0;         // first K half this warp converts
    const int h1 = (wps == 8) ? h0 + 1 : 2;
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // wr: weight slot of the stage; ar: its A slot; dr: the done barrier of the
    // stage NB earlier, the last one that used the same A slot (phase of lap -1,
    // which a fresh barrier reports complete, for the first NB stages)
    Ring wr, ar, dr;
    wr.idx = ar.idx = set;
    dr.idx = set - NB + NB2;
    dr.phase = 1u;
    int g0 = 0;
    bool ok = true;
    // A-slot wait (first half) and the sparse-MMA store of one half: kept values to
    // columns 16h .. 16h+15 of the A slot, the position words of MMAs 2h and 2h+1 to
    // columns 32 + 16h and 40 + 16h
    auto sparse_store = [&](int half, int hfirst, const uint2& pos, const uint32_t (&vals)[16]) -> bool {
      if (NB2 != NB && half == hfirst) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done + dr.idx), dr.phase, abort_flag, 512));
        if (!ok) return false;
        tc_fence_after();
      }
      const uint32_t ta = tmem + lane_base + a_col0 + static_cast<uint32_t>(ar.idx * 64);
      tmem_st_32x32b_x16(ta + static_cast<uint32_t>(16 * half), vals);
      tmem_st_32x32b_x1(ta + 32u + static_cast<uint32_t>(16 * half), pos.x);
      tmem_st_32x32b_x1(ta + 40u + static_cast<uint32_t>(16 * half), pos.y);
      return true;
    };
    for (int i = item0; i < n_items && ok; i += item_step) {
      WorkItem it;
      decode_item<PAIR>(p, nch, i, rank, it);
      const int n_st = it.ks1 - it.ks0;
      for (int g = first_own(g0, set, DS); g < g0 + n_st;
           g += DS, wr.step(DS, NW), ar.step(DS, NB), dr.step(DS, NB2)) {
        // weights and token tile landed
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(wfull + wr.idx), wr.phase, abort_flag, 512));
        if (!ok) break;
        tc_fence_after();
        const uint32_t ws_a = smem_u32(wring + wr.idx * wslot);  // the stage's weight slot (shared window)
        for (int half = h0; half < h1; ++half) {
          const bool last = half + 1 == h1;  // the weight slot is released after the last half's loads
          uint32_t out[32];
          if (INT4) {
            uint4 pk[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) pk[c] = lds_u128(ws_a + ((2 * half + c) * 128 + row) * 16);
            const uint32_t sbits = lds_u16(ws_a + 8192 + row * 2);
            const uint32_t zp = (KIND == kQ4Z) ? lds_u8(ws_a + 8448 + row) : 8u;
            __syncwarp();
            if (last && lane == 0) mbar_arrive(smem_u32(wempty + wr.idx));
            if (PG) {
              dequant_int4_raw_half(pk, out);  // the epilogue applies scale and zero point
            } else {
              // two 16-column pieces, each converted and stored in turn (16 live
              // registers of converted values instead of 32)
              uint32_t bias_bits, m64z;
              int4_zp_constants(zp, bias_bits, m64z);
              const uint32_t s2bits = int4_scale_pair<BF16S>(sbits);
              const uint32_t ta = tmem + lane_base + a_col0 + static_cast<uint32_t>(ar.idx * 64 + 32 * half);
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                uint32_t o16[16];
                dequant_int4_chunk(pk[c], bias_bits, m64z, s2bits, o16);
                if (c == 0 && NB2 != NB && half == h0) {
                  ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done + dr.idx), dr.phase, abort_flag, 512));
                  if (!ok) break;
                  tc_fence_after();
                }
                tmem_st_32x32b_x16(ta + 16u * c, o16);
              }
              if (!ok) break;
              continue;
            }
          } else if (KIND == kQ4S) {
            const uint4 pk = lds_u128(ws_a + (half * 128 + row) * 16);
            const uint2 pos = lds_u64(ws_a + 4096 + (half * 128 + row) * 8);
            const uint32_t sbits = lds_u16(ws_a + 6144 + row * 2);
            __syncwarp();
            if (last && lane == 0) mbar_arrive(smem_u32(wempty + wr.idx));
            uint32_t vals[16];
            dequant_int4_24_vals_half<BF16S>(pk, sbits, vals);
            if (!sparse_store(half, h0, pos, vals)) break;
            continue;
          } else if (KIND == kQ8S || KIND == kQ8SG) {
            uint4 pk[2];
#pragma unroll
            for (int c = 0; c < 2; ++c)
              pk[c] = lds_u128(ws_a + (half * 128 + row) * 32 + 16 * c);
            const uint2 pos = lds_u64(ws_a + 8192 + (half * 128 + row) * 8);
            const uint32_t sbits = (KIND == kQ8SG) ? lds_u16(ws_a + 10240 + row * 2) : 0u;
            __syncwarp();
            if (last && lane == 0) mbar_arrive(smem_u32(wempty + wr.idx));
            uint32_t vals[16];
            dequant_int8_24_vals_half<KIND == kQ8SG, BF16S>(pk, sbits, vals);
            if (!sparse_store(half, h0, pos, vals)) break;
            continue;
          } else {
            uint4 pk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) pk[c] = lds_u128(ws_a + ((4 * half + c) * 128 + row) * 16);
            const uint32_t sbits = (KIND == kQ8G) ? lds_u16(ws_a + 16384 + row * 2) : 0u;
            __syncwarp();
            if (last && lane == 0) mbar_arrive(smem_u32(wempty + wr.idx));
            dequant_int8_half<KIND == kQ8G, BF16S>(pk, sbits, out);
          }
          // the A slot is free once the MMAs of the stage NB earlier completed; with
          // token-tile and A rings of one depth the token tile's arrival implied it
          // (the producer waited for the same barrier phase before copying it)
          if (NB2 != NB && half == h0) {
            ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done + dr.idx), dr.phase, abort_flag, 512));
            if (!ok) break;
            tc_fence_after();
          }
          const uint32_t ta = tmem + lane_base + a_col0 + static_cast<uint32_t>(ar.idx * 64 + 32 * half);
          tmem_st_32x32b_x32<0>(ta, out);
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // (a pair's A barriers live in the even CTA and count both CTAs' sets)
          if (PAIR)
            mbar_arrive_remote(map_to_rank(smem_u32(afull + ar.idx), 0));
          else
            mbar_arrive(smem_u32(afull + ar.idx));
        }
      }
      g0 += n_st;
    }
    if (!ok && lane == 0) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue warpgroup
    const int q = warp;
    const int row = q * 32 + lane;  // weight row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int itn = 0, g0 = 0;
    bool ok = true;
    if (PG) {
      // Per-group scaling: every stage's sum D (fp32, its own D slot) becomes
      //   acc += s_g * (D - C_g[token]),
      // s_g the row's group scale, C_g the token row's correction for the raw
      // magic-number halves (see the gather).  Reading D releases the stage's A
      // slot to the issuer (the afull barrier also counts these 4 arrivals); the
      // first use of each slot is released here at the start.
      //
      // Scales and corrections reach shared memory by per-thread async copies,
      // for segments of kPgSeg stages of the CTA's stage sequence, two segments
      // ahead, into buffers private to the warp (so a wait_group and a
      // __syncwarp order them; no barrier across warps).
      if (lane == 0)
        for (int j = 0; j < NB; ++j) mbar_arrive(smem_u32(afull + j));
      uint8_t* wbuf = reinterpret_cast<uint8_t*>(wfull) + kBarrierBytes + q * 2 * kPgWarpBuf;
      struct Seg {
        int i, s0, n;  // item, first stage within it, stages (0: past the last item)
        WorkItem it;
      };
      auto seg_first = [&](Seg& sg) {
        sg.i = item0;
        sg.s0 = 0;
        if (sg.i < n_items) decode_item<PAIR>(p, nch, sg.i, rank, sg.it);
        sg.n = sg.i < n_items ? min(kPgSeg, sg.it.ks1 - sg.it.ks0) : 0;
      };
      auto seg_next = [&](Seg& sg) {
        if (sg.n == 0) return;
        sg.s0 += sg.n;
        if (sg.s0 == sg.it.ks1 - sg.it.ks0) {
          sg.i += item_step;
          sg.s0 = 0;
          if (sg.i >= n_items) {
            sg.n = 0;
            return;
          }
          decode_item<PAIR>(p, nch, sg.i, rank, sg.it);
        }
        sg.n = min(kPgSeg, sg.it.ks1 - sg.it.ks0 - sg.s0);
      };
      // segment -> buffer b: 4 x n pieces of 16 bytes each of scales (the warp's
      // 64 bytes of a stage's 256) and of corrections (a stage's 16 fp32)
      auto seg_fetch = [&](const Seg& sg, int b) {
        uint8_t* dst = wbuf + b * kPgWarpBuf;
        const uint8_t* sbase = p.w +
                               ((static_cast<int64_t>(sg.it.e) * p.n_tiles + sg.it.tile) * p.k_groups + sg.it.ks0 + sg.s0) *
                                   static_cast<int64_t>(p.stage_bytes) +
                               8192 + q * 64;
        const float* cbase = p.pg_corr + static_cast<int64_t>(sg.it.ks0 + sg.s0) * p.pg_cap + sg.it.row0;
        for (int j = lane; j < 4 * sg.n; j += 32) {
          const int st = j >> 2, part = j & 3;
          cp_async_16(smem_u32(dst + st * 64 + part * 16), sbase + static_cast<int64_t>(st) * p.stage_bytes + part * 16);
          cp_async_16(smem_u32(dst + kPgSeg * 64 + st * 64 + part * 16), cbase + static_cast<int64_t>(st) * p.pg_cap + 4 * part);
        }
        cp_async_commit();
      };
      Seg use, fetch;
      seg_first(use);
      fetch = use;
      seg_fetch(fetch, 0);
      seg_next(fetch);
      seg_fetch(fetch, 1);
      seg_next(fetch);
      Ring ar, dn;
      int ub = 0;
      float acc[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[c] = 0.0f;
      while (use.n > 0 && ok) {
        cp_async_wait_group<1>();
        __syncwarp();
        const uint8_t* buf = wbuf + ub * kPgWarpBuf;
        for (int st = 0; st < use.n; ++st, ar.step(1, NB), dn.step(1, NB2)) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done + dn.idx), dn.phase, abort_flag, 32));
          if (!ok) break;
          tc_fence_after();
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_base + static_cast<uint32_t>(p.d_col0 + ar.idx * 16), v);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(afull + ar.idx));
          // the f16 value of the group scale that the standard path multiplies by
          const uint32_t buf_a = smem_u32(buf);
          const uint16_t sb = static_cast<uint16_t>(lds_u16(buf_a + st * 64 + 2 * lane));
          const float sg = BF16S ? __half2float(__float2half_rn(__uint_as_float(static_cast<uint32_t>(sb) << 16)))
                                 : __half2float(__ushort_as_half(sb));
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 cb = lds_u128(buf_a + kPgSeg * 64 + st * 64 + 16 * c);
            const float4 cv = make_float4(__uint_as_float(cb.x), __uint_as_float(cb.y), __uint_as_float(cb.z),
                                          __uint_as_float(cb.w));
            acc[4 * c] = fmaf(sg, __uint_as_float(v[4 * c]) - cv.x, acc[4 * c]);
            acc[4 * c + 1] = fmaf(sg, __uint_as_float(v[4 * c + 1]) - cv.y, acc[4 * c + 1]);
            acc[4 * c + 2] = fmaf(sg, __uint_as_float(v[4 * c + 2]) - cv.z, acc[4 * c + 2]);
            acc[4 * c + 3] = fmaf(sg, __uint_as_float(v[4 * c + 3]) - cv.w, acc[4 * c + 3]);
          }
        }
        if (!ok) break;
        // every lane is done with this buffer: refill it two segments ahead
        __syncwarp();
        if (fetch.n > 0) {
          seg_fetch(fetch, ub);
          seg_next(fetch);
        } else {
          cp_async_commit();  // an empty group keeps the wait_group count in step
        }
        ub ^= 1;
        if (use.s0 + use.n == use.it.ks1 - use.it.ks0) {
          const float4* cs4 = reinterpret_cast<const float4*>(p.col_scale + use.it.row0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 v4 = __ldg(cs4 + c);
            acc[4 * c] *= v4.x;
            acc[4 * c + 1] *= v4.y;
            acc[4 * c + 2] *= v4.z;
            acc[4 * c + 3] *= v4.w;
          }
          epilogue_store(p, use.it, 0, row, lane, acc);
#pragma unroll
          for (int c = 0; c < 16; ++c) acc[c] = 0.0f;
        }
        seg_next(use);
      }
      // no copy of this thread may still be in flight when the CTA exits
      cp_async_wait_group<0>();
    }
    for (int i = PG ? n_items : item0; i < n_items && ok; i += item_step) {
      WorkItem it;
      decode_item<PAIR>(p, nch, i, rank, it);
      const int b = (ACCB == 2) ? (itn & 1) : 0;
      const uint32_t use = (ACCB == 2) ? (itn >> 1) : itn;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(accfull + b), use & 1u, abort_flag, 512));
      if (!ok) break;
      tc_fence_after();
      // issuer j took the item's stages g0 + n with (g0 + n) % NI == j
      const int n_st = it.ks1 - it.ks0;
      bool has[kMaxIssuers];
#pragma unroll
      for (int j = 0; j < kMaxIssuers; ++j) has[j] = j < NI && first_own(g0, j, NI) < g0 + n_st;
      g0 += n_st;
      const float rs = (KIND != kQ8 && KIND != kQ8S)
                           ? 1.0f
                           : __ldg(p.row_scale + (static_cast<int64_t>(it.e) * p.n_tiles + it.tile) * kTileRows + row);
      for (int c0 = 0; c0 < it.nrows; c0 += 16) {
        float f[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) f[c] = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxIssuers; ++j) {
          if (!has[j]) continue;
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_base + static_cast<uint32_t>((j * ACCB + b) * T + c0), v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; ++c) f[c] += __uint_as_float(v[c]);
        }
        if (c0 + 16 >= it.nrows) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR)
              mbar_arrive_remote(map_to_rank(smem_u32(accempty + b), 0));
            else
              mbar_arrive(smem_u32(accempty + b));
          }
        }
        const float4* cs4 = reinterpret_cast<const float4*>(p.col_scale + it.row0 + c0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 v4 = __ldg(cs4 + c);
          f[4 * c] *= rs * v4.x;
          f[4 * c + 1] *= rs * v4.y;
          f[4 * c + 2] *= rs * v4.z;
          f[4 * c + 3] *= rs * v4.w;
        }
        if (!it.phantom) epilogue_store(p, it, c0, row, lane, f);
      }
      ++itn;
    }
    if (!ok && lane == 0) raise_abort(reinterpret_cast<volatile int*>(abort_flag), p.status);
  }

  // ------------------------------------------------------------ teardown
  // (on CTA pairs no remote arrive and no pair MMA touches either CTA after the
  // cluster barrier)
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
}

template <int KIND, bool BF16S, bool PAIR = false>
cudaError_t launch_gemm_t(const GemmParams& p, int grid, cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(p);
  cudaError_t err = cudaFuncSetAttribute(qmoe_gemm_kernel<KIND, BF16S, PAIR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  if (!PAIR) return launch_kernel(qmoe_gemm_kernel<KIND, BF16S, PAIR>, dim3(grid), dim3(kGemmThreads), smem, stream, true, p);
  // clusters of 2 CTAs (an even grid)
  if (grid % 2 != 0 || p.pair == 0) return cudaErrorInvalidValue;
  return launch_kernel_cluster(qmoe_gemm_kernel<KIND, BF16S, PAIR>, dim3(grid), dim3(kGemmThreads), smem, stream, true,
                               2u, p);
}

}  // namespace qmoe
