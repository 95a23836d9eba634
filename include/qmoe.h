/*
 * qmoe.h - C ABI of libqmoe, a GB300 (sm_103a) fused mixture-of-experts layer
 * whose expert weights are weight-only quantized (W4A16 GPTQ-style int4 with
 * group scales and optional act-order, or W8A16 per-column int8).
 *
 * The layer computed by qmoe_forward, for tokens m = 0..M-1 and top-k slots j:
 *
 *     e     = topk_ids[m, j]
 *     h     = W13_e · x[m]                  (W13_e = [gate_e ; up_e], 2I x H)
 *     t     = SiLU(h[0:I]) * h[I:2I]
 *     y     = W2_e · t                      (W2_e: H x I)
 *     out[m] = sum_j topk_weights[m, j] * y
 *
 * with the expert matrices dequantized on the fly:
 *     int4:  W[n, k] = (q[n, k] - 8) * s[g(k), n],  g(k) = g_idx[k] (act-order) or k / 128
 *     int8:  W[n, k] = q[n, k] * s[n]
 *
 * Sources (web pages on this method):
 *   "Marlin moe integration" (nm-vllm pull request): the fused MoE kernel takes
 *     already-quantized INT4 weights and scales on the hot path, quantization
 *     lives in test utilities; GPTQ 4-bit group-128 checkpoints with and without
 *     act-order; moe_align_block_size with block size 16; scales normalised to
 *     the half type on load.
 *   "[Kernel] W8A16 Int8 inside FusedMoE" (vLLM pull request): symmetric
 *     per-column, per-expert int8 cast to FP16/BF16 before the matmul; explicit
 *     W8A16 vs W8A8 naming.
 *   "Add GPTQ Marlin 2:4 sparse structured support": group 128 or channel-wise,
 *     4 or 8 bits.
 *   "[WIP] AWQ Faster Kernels" (vLLM issue): the batch dimension must reach the
 *     kernel chooser (so M is always an explicit argument here); packed-dimension
 *     bugs in weight loading (so the packing dimension is documented below).
 *
 * Conventions for every entry point:
 *   - No function allocates memory, and none synchronises the stream except
 *     qmoe_read_device_status.  All device work is enqueued on `stream`
 *     (a cudaStream_t passed as void*; NULL is the legacy default stream) and
 *     runs asynchronously.  Every buffer is owned by the caller.
 *   - Arguments are validated before anything is launched; on any error
 *     nothing is launched and the status says why.  No exception crosses the ABI.
 *   - Device pointers must be device (or managed) memory of the current CUDA
 *     device; a pointer of another device gives QMOE_ERR_DEVICE_MISMATCH.
 *   - Faults the host cannot see (a top-k id outside [0, E), a kernel wait that
 *     ran past its time limit) are recorded in the workspace and read back with
 *     qmoe_read_device_status.
 *   - The library is stateless apart from a per-device cache of the SM count
 *     (and, for qmoe_forward_noalloc, of its scratch array's address); calls
 *     are thread-safe.
 */
#ifndef QMOE_H_
#define QMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMOE_ABI_VERSION 2

typedef enum {
  QMOE_OK = 0,
  QMOE_ERR_INVALID_ARG = 1,     /* bad size, null pointer, misalignment, bad enum */
  QMOE_ERR_UNSUPPORTED = 2,     /* valid but not implemented (shape, group size, dtype combo) */
  QMOE_ERR_DEVICE_MISMATCH = 3, /* a pointer is not device memory of the current device */
  QMOE_ERR_WORKSPACE = 4,       /* workspace null or smaller than qmoe_workspace_size */
  QMOE_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed */
  QMOE_ERR_TIMEOUT = 6,         /* device: a pipeline wait ran past its limit and the kernel gave up */
  QMOE_ERR_BAD_EXPERT_ID = 7    /* device: a top-k id outside [0, E); that pair was dropped */
} qmoe_status;

typedef enum {
  QMOE_INT4_GROUP = 1,    /* 4-bit codes 0..15, zero point 8, one scale per 128 input channels
                             (group_size 128) or per output feature (group_size -1) */
  QMOE_INT8_PER_COL = 2,  /* signed 8-bit codes, one float32 scale per output feature */
  QMOE_INT4_GROUP_ZP = 3, /* 4-bit codes 0..15 with a zero point 0..15 and a scale per group
                             (128 input channels, or all of them with group_size -1) */
  QMOE_INT8_GROUP = 4,    /* signed 8-bit codes, one scale per 128 input channels */
  QMOE_INT4_GROUP_24 = 5, /* as QMOE_INT4_GROUP, 2:4 sparse along K: in every aligned group of
                             4 input channels at most 2 codes differ from 8 (value 0); only
                             those 2 codes and their positions are stored */
  QMOE_INT8_24 = 6        /* signed 8-bit codes, 2:4 sparse along K (at most 2 non-zero codes in
                             every aligned group of 4 input channels; the 2 kept codes and their
                             positions are stored), with one float32 scale per output feature
                             (group_size -1) or one scale of the activation type per 128 input
                             channels (group_size 128) */
} qmoe_quant_type;

typedef enum { QMOE_F16 = 1, QMOE_BF16 = 2, QMOE_F32 = 3 } qmoe_dtype;

/*
 * One MoE layer, weights already packed by one of the qmoe_pack_* functions.
 * All pointers are device memory owned by the caller and must stay valid
 * while work that uses them is in flight.
 *
 *   E, H, I      experts, hidden size, expert intermediate size.
 *                Constraints: 1 <= E <= 1024; H % 128 == 0; I % 128 == 0.
 *   group_size   QMOE_INT4_GROUP / QMOE_INT4_GROUP_ZP / QMOE_INT4_GROUP_24 /
 *                QMOE_INT8_24: 128 or -1 (channel-wise); QMOE_INT8_PER_COL: -1;
 *                QMOE_INT8_GROUP: 128.  The 2:4-sparse formats take no
 *                act-order permutation.
 *   qt           quantization type.
 *   act_dtype    F16 or BF16: type of x and out (the MMAs run in f16).
 *   scale_dtype  int4 and grouped int8 (also 2:4-sparse int8 with group_size
 *                128): must equal act_dtype (scales are normalised to the
 *                activation type when packed); per-column int8 and
 *                channel-wise 2:4-sparse int8: F32.
 *   w13, w2      packed expert weights (sizes: qmoe_packed_bytes), 256-byte aligned.
 *   s13, s2      per-column int8 and channel-wise 2:4-sparse int8 only:
 *                float32 scales packed by qmoe_pack_int8 / qmoe_pack_int8_24
 *                ([E, 2I] in packed row order, [E, H]); NULL otherwise (the
 *                other formats keep their scales and zero points inside the
 *                packed weights).
 *   perm13       int4 act-order only (group_size 128): int32 [E, H] written
 *                by qmoe_pack_int4 / qmoe_pack_int4_zp (hidden channel of
 *                each sorted K position); NULL otherwise.  With act-order H is
 *                at most 65536 (QMOE_ERR_UNSUPPORTED otherwise).
 *                Act-order of W2 needs no runtime table: it is folded into the
 *                row order of the packed W13.
 */
typedef struct {
  int32_t E, H, I;
  int32_t group_size;
  qmoe_quant_type qt;
  qmoe_dtype act_dtype;
  qmoe_dtype scale_dtype;
  const void* w13;
  const void* w2;
  const float* s13;
  const float* s2;
  const int32_t* perm13;
} qmoe_layer;

/*
 * Optional tuning knobs (zero = automatic).  Results are identical up to
 * floating-point summation order whatever the knobs say.
 *   split1, split2  split-K factor of the gate/up and down GEMMs (1..64).
 *   token_tile      largest number of token rows one GEMM work item carries
 *                   (multiple of 16, 16..256).
 *   issuers         warps issuing the GEMMs' tensor-core MMAs (1..3), each
 *                   with its own TMEM accumulator; the automatic choice is 2
 *                   for token tiles of up to 64 rows, else 1.  The automatic
 *                   token tile is the power of two from 16 to 128 at least 1.5
 *                   times the mean number of pairs per expert, and at least 32
 *                   when E >= 16 * top_k and M >= 32 (an expert's pairs can
 *                   reach M, E / top_k times the mean).
 * Other values, or an issuer count whose accumulators leave too little tensor
 * memory for the pipeline, give QMOE_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t split1;
  int32_t split2;
  int32_t token_tile;
  /* Test hook for the device-side failure path (0 = off).  1: in the gate/up
   * GEMM, CTA 0 arms its first pipeline stage without issuing the copies that
   * complete it, so its consumers wait on a phase that never completes; the
   * bounded waits give up after about a second, record QMOE_ERR_TIMEOUT and the
   * kernel exits with the CUDA context intact (the output is then garbage). */
  int32_t fault_injection;
  int32_t issuers;
  /* Depth of the GEMMs' shared-memory token-tile ring as a multiple (1..3) of
   * the TMEM A ring (0: automatic, 2 where shared memory leaves the weight ring
   * at least 8 slots, else 1).  A value whose ring does not fit gives
   * QMOE_ERR_INVALID_ARG. */
  int32_t token_ring;
  /* Dequant warp sets of the GEMMs: 2 (8 warps each, half a stage row per
   * warp) or 4 (4 warps each, whole rows per warp); 0: automatic (4 wherever
   * the rings allow it).  4 needs a token-tile ring that is a multiple of 4
   * and at least 4 TMEM A slots (QMOE_ERR_INVALID_ARG otherwise). */
  int32_t dq_sets;
  /* L2 policy of the GEMMs' weight copies: 0 automatic (evict-normal when an
   * expert has more pairs than one token tile, so that the chunks that share
   * a weight tile find it in L2; evict-first otherwise), 1 evict-normal,
   * 2 evict-first.  Other values give QMOE_ERR_INVALID_ARG. */
  int32_t weight_l2;
  /* Symmetric int4 with 16-row token tiles: 0 automatic (off), 1 on, 2 off.  On,
   * the dequant warps hand the tensor core the raw magic-number halves of the
   * codes (1024 + q and 1024 + 16 q against tokens pre-divided by 16) and the
   * epilogue applies each 128-channel group's scale and zero point in fp32, per
   * pipeline stage.  1 where it does not apply gives QMOE_ERR_INVALID_ARG. */
  int32_t int4_group_epilogue;
  /* Top-k reduction (summing each token's expert outputs and K splits):
   * 0 automatic (a separate kernel), 1 in the down GEMM's epilogue (the warp
   * that completes a token's arrival count sums its partials; one launch
   * fewer, slower on GB300), 2 a separate kernel.  Both sum in the same fixed
   * order (results are bit-identical).  Other values give QMOE_ERR_INVALID_ARG. */
  int32_t topk_reduce;
  /* GEMMs on CTA pairs: 0 automatic, 1 on, 2 off.  On, each GEMM runs as
   * clusters of two CTAs on two SMs: one M = 256 tensor-core MMA (tcgen05
   * cta_group::2) covers both CTAs' 128-row weight tiles, and each CTA copies
   * only half of the token tile's rows into its shared memory.  Symmetric int4
   * (QMOE_INT4_GROUP) and QMOE_INT8_PER_COL only, not with topk_reduce = 1 or
   * int4_group_epilogue = 1 (QMOE_ERR_INVALID_ARG otherwise).  Automatic (with
   * token_ring automatic): on where shared memory leaves a single CTA a
   * token-tile ring of one A-ring depth or fewer than 8 weight slots (large
   * token tiles; 64-row tiles of int8). */
  int32_t cta_pair;
  int32_t reserved[5];  /* must be zero */
} qmoe_options;

/* ------------------------------------------------------------------------ */
/* Weight packing (host memory in, host memory out; off the hot path).       */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of one packed matrix for all E experts: W13 is (rows = 2I, K = H),
 * W2 is (rows = H, K = I).  Returns 0 for an unsupported combination.
 * Per 128 x 128 block: QMOE_INT4_GROUP 8448 (group_size 128 or -1),
 * QMOE_INT4_GROUP_ZP 8576 (group_size 128 or -1), QMOE_INT4_GROUP_24 6400
 * (group_size 128 or -1), QMOE_INT8_PER_COL 16384 (group_size -1),
 * QMOE_INT8_GROUP 16640 (group_size 128), QMOE_INT8_24 10240 (group_size -1)
 * or 10496 (group_size 128); times E * (rows/128) * (K/128).
 */
size_t qmoe_packed_bytes(qmoe_quant_type qt, int32_t E, int32_t rows, int32_t K, int32_t group_size);

/*
 * Pack int4 GPTQ-style weights ("Marlin moe integration": the kernel receives
 * already-quantized INT4 weights and scales; GPTQ group 128, act-order).
 * Canonical inputs (host, row-major, one code per byte, packing dimension = K):
 *   q13 uint8 [E, 2I, H] codes 0..15 (rows 0..I-1 gate, I..2I-1 up)
 *   s13 uint16 [E, H/128, 2I] scale bit patterns of scale_dtype (f16 or bf16)
 *   g13 int32 [E, H] group of each hidden channel, or NULL (group = k/128)
 *   q2  uint8 [E, H, I],  s2 uint16 [E, I/128, H],  g2 int32 [E, I] or NULL
 * Outputs (host): w13_packed, w2_packed (qmoe_packed_bytes each) and, when
 * g13 != NULL, perm13_out int32 [E, H]; perm13_out is ignored when g13 == NULL.
 * Act-order requires every group to hold exactly 128 channels (as GPTQ's
 * act-order produces); otherwise QMOE_ERR_UNSUPPORTED.  Codes above 15 give
 * QMOE_ERR_INVALID_ARG.  group_size -1 is one scale per output feature over
 * all of K ("Add GPTQ Marlin 2:4 sparse structured support" lists group 128
 * or -1, channel-wise): s13 is then [E, 1, 2I] and s2 [E, 1, H], and g13 /
 * g2 must be NULL (QMOE_ERR_UNSUPPORTED otherwise).
 */
qmoe_status qmoe_pack_int4(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                           const uint8_t* q13, const uint16_t* s13, const int32_t* g13,
                           const uint8_t* q2, const uint16_t* s2, const int32_t* g2,
                           void* w13_packed, void* w2_packed, int32_t* perm13_out);

/* Exact inverse of qmoe_pack_int4 given the same g13 / g2 (round-trip checks). */
qmoe_status qmoe_unpack_int4(int32_t E, int32_t H, int32_t I, int32_t group_size,
                             const void* w13_packed, const void* w2_packed,
                             const int32_t* g13, const int32_t* g2,
                             uint8_t* q13, uint16_t* s13, uint8_t* q2, uint16_t* s2);

/*
 * Pack asymmetric int4 with one zero point per group ("[WIP] AWQ Faster
 * Kernels": AWQ checkpoints store per-group zero points):
 * W[n, k] = (q[n, k] - z[g(k), n]) * s[g(k), n].  Arguments as for
 * qmoe_pack_int4 plus z13 uint8 [E, H/128, 2I] and z2 uint8 [E, I/128, H]
 * (zero points 0..15; [E, 1, *] with group_size -1).  Zero points above 15
 * give QMOE_ERR_INVALID_ARG.  The layer's qt is QMOE_INT4_GROUP_ZP.
 */
qmoe_status qmoe_pack_int4_zp(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const uint8_t* q13, const uint16_t* s13, const uint8_t* z13, const int32_t* g13,
                              const uint8_t* q2, const uint16_t* s2, const uint8_t* z2, const int32_t* g2,
                              void* w13_packed, void* w2_packed, int32_t* perm13_out);

/* Exact inverse of qmoe_pack_int4_zp given the same g13 / g2. */
qmoe_status qmoe_unpack_int4_zp(int32_t E, int32_t H, int32_t I, int32_t group_size,
                                const void* w13_packed, const void* w2_packed,
                                const int32_t* g13, const int32_t* g2,
                                uint8_t* q13, uint16_t* s13, uint8_t* z13,
                                uint8_t* q2, uint16_t* s2, uint8_t* z2);

/*
 * Pack symmetric int8 with one scale per 128 input channels ("Add GPTQ Marlin
 * 2:4 sparse structured support" lists 8-bit with group 128):
 * W[n, k] = q[n, k] * s[k / 128, n].  Canonical inputs (host):
 *   q13 int8 [E, 2I, H], s13 uint16 [E, H/128, 2I] scale bit patterns of
 *   scale_dtype (f16 or bf16); q2 int8 [E, H, I], s2 uint16 [E, I/128, H].
 * Outputs (host): w13_packed, w2_packed (the scales live inside the packed
 * blocks).  Codes of -128 give QMOE_ERR_INVALID_ARG.  The layer's qt is
 * QMOE_INT8_GROUP with group_size 128.
 */
qmoe_status qmoe_pack_int8_group(int32_t E, int32_t H, int32_t I, qmoe_dtype scale_dtype,
                                 const int8_t* q13, const uint16_t* s13, const int8_t* q2, const uint16_t* s2,
                                 void* w13_packed, void* w2_packed);

/*
 * Pack 2:4-sparse int4 ("Add GPTQ Marlin 2:4 sparse structured support":
 * 4-bit, group 128 or channel-wise, 2:4 structured sparsity).  Canonical
 * inputs (host) as for qmoe_pack_int4 without g_idx: q13 uint8 [E, 2I, H] and
 * q2 uint8 [E, H, I] dense codes 0..15 with zero point 8, where every aligned
 * group of 4 consecutive input channels holds at most 2 codes other than 8;
 * s13 uint16 [E, H/128 (or 1), 2I], s2 uint16 [E, I/128 (or 1), H] scale bit
 * patterns of scale_dtype.  Per group of 4 the packer keeps the channels whose
 * code is not 8, padded with the lowest remaining channels, as 2 codes and 2
 * two-bit positions.  Outputs (host): w13_packed, w2_packed.  A group with
 * more than 2 codes other than 8, or a code above 15, gives
 * QMOE_ERR_INVALID_ARG.  The layer's qt is QMOE_INT4_GROUP_24.
 */
qmoe_status qmoe_pack_int4_24(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const uint8_t* q13, const uint16_t* s13, const uint8_t* q2, const uint16_t* s2,
                              void* w13_packed, void* w2_packed);

/* Exact inverse of qmoe_pack_int4_24 (dense codes, 8 at the pruned channels). */
qmoe_status qmoe_unpack_int4_24(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                                const void* w2_packed, uint8_t* q13, uint16_t* s13, uint8_t* q2, uint16_t* s2);

/*
 * Pack 2:4-sparse int8 ("Add GPTQ Marlin 2:4 sparse structured support":
 * 8-bit, group 128 or channel-wise, 2:4 structured sparsity).  Canonical
 * inputs (host): q13 int8 [E, 2I, H] and q2 int8 [E, H, I] dense codes
 * -127..127 where every aligned group of 4 consecutive input channels holds
 * at most 2 non-zero codes.  group_size -1 (scale_dtype QMOE_F32): s13 float
 * [E, 2I], s2 float [E, H], one scale per output feature, W = q * s[n];
 * outputs s13_packed float [E, 2I] (packed row order) and s2_packed float
 * [E, H] as for qmoe_pack_int8.  group_size 128 (scale_dtype F16 or BF16):
 * s13 uint16 [E, H/128, 2I], s2 uint16 [E, I/128, H] scale bit patterns,
 * W = q * s[k/128, n], kept inside the packed blocks (s13_packed / s2_packed
 * may be NULL).  Per group of 4 the packer keeps the non-zero codes, padded
 * with the lowest remaining channels.  More than 2 non-zero codes in a group,
 * or a code of -128, gives QMOE_ERR_INVALID_ARG.  The layer's qt is
 * QMOE_INT8_24.
 */
qmoe_status qmoe_pack_int8_24(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const int8_t* q13, const void* s13, const int8_t* q2, const void* s2,
                              void* w13_packed, float* s13_packed, void* w2_packed, float* s2_packed);

/* Exact inverse of qmoe_pack_int8_24 (dense codes, 0 at the pruned channels; s13 / s2 as packed). */
qmoe_status qmoe_unpack_int8_24(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                                const float* s13_packed, const void* w2_packed, const float* s2_packed,
                                int8_t* q13, void* s13, int8_t* q2, void* s2);

/* Exact inverse of qmoe_pack_int8_group. */
qmoe_status qmoe_unpack_int8_group(int32_t E, int32_t H, int32_t I, const void* w13_packed, const void* w2_packed,
                                   int8_t* q13, uint16_t* s13, int8_t* q2, uint16_t* s2);

/*
 * Pack W8A16 per-column int8 ("[Kernel] W8A16 Int8 inside FusedMoE":
 * symmetric per-column, per-expert int8).  Canonical inputs (host):
 *   q13 int8 [E, 2I, H], s13 float [E, 2I]; q2 int8 [E, H, I], s2 float [E, H].
 * Outputs (host): w13_packed, w2_packed, s13_packed float [E, 2I] (packed row
 * order), s2_packed float [E, H].  Codes of -128 give QMOE_ERR_INVALID_ARG.
 */
qmoe_status qmoe_pack_int8(int32_t E, int32_t H, int32_t I,
                           const int8_t* q13, const float* s13, const int8_t* q2, const float* s2,
                           void* w13_packed, float* s13_packed, void* w2_packed, float* s2_packed);

/* Exact inverse of qmoe_pack_int8. */
qmoe_status qmoe_unpack_int8(int32_t E, int32_t H, int32_t I,
                             const void* w13_packed, const float* s13_packed,
                             const void* w2_packed, const float* s2_packed,
                             int8_t* q13, float* s13, int8_t* q2, float* s2);

/* ------------------------------------------------------------------------ */
/* moe_align_block_size                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Group the P = M*top_k token-expert pairs by expert and pad each group to a
 * multiple of `block` ("Marlin moe integration": moe_align_block_size_kernel,
 * block size 16 tied to the kernel tile).  Deterministic and stable:
 *   sorted_ids      int32 [capacity]: experts in ascending id, each expert's
 *                   pair indices p = m*top_k + j ascending, padded with P;
 *                   the tail past the padded total also holds P.
 *   expert_ids      int32 [ceil(capacity/block)]: expert of each block; -1
 *                   for blocks past the padded total.
 *   num_post_padded int32 [1]: padded total (a multiple of block).
 * Device inputs: topk_ids int32 [M, top_k].  Requirements: 1 <= E <= 1024,
 * 1 <= block <= 256, capacity >= M*top_k + E*(block-1), M*top_k < 2^31.
 * Ids outside [0, E) are dropped (not placed).  M == 0 is valid.
 */
qmoe_status qmoe_moe_align(const int32_t* topk_ids, int64_t M, int32_t top_k, int32_t E, int32_t block,
                           int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                           int64_t capacity, void* stream);

/* ------------------------------------------------------------------------ */
/* Forward                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Workspace bytes qmoe_forward needs for this layer, M and top_k (0 on invalid
 * input).  The batch size M is an explicit argument of every sizing and launch
 * call ("[WIP] AWQ Faster Kernels", discussion: the kernel choice depends on
 * the number of tokens, which must reach the kernel chooser).  The workspace
 * holds the moe_align output ("Marlin moe integration", review thread), the
 * gathered activations, the intermediate and the split-K partial sums.
 */
size_t qmoe_workspace_size(const qmoe_layer* layer, int64_t M, int32_t top_k);
size_t qmoe_workspace_size_ex(const qmoe_layer* layer, int64_t M, int32_t top_k, const qmoe_options* opts);

/*
 * The launch plan qmoe_forward_ex would use (host only; no device access when
 * num_sms > 0).  Fields: token_tile (token rows per GEMM work item), issuers
 * (MMA-issuing warps per CTA), acc_bufs (TMEM accumulators per issuer),
 * split1 / split2 (split-K of the gate/up and down GEMMs), w_stages (packed-
 * weight ring depth), ab_stages (TMEM A ring depth), b_stages (token-tile ring
 * depth, a multiple of ab_stages), dq_sets (dequant warp sets), cta_pair (1: the
 * gate/up GEMM runs on CTA pairs; the ring fields describe that GEMM),
 * cta_pair_down (1: the down GEMM runs on CTA pairs too; automatic plans keep it
 * on single CTAs when its K spans fewer than 32 stages of 128), stage_bytes
 * (packed bytes per 128 x 128 block), workspace_bytes.  num_sms: the GPU's
 * SM count the plan is sized for (0: the current device's).  Errors as
 * qmoe_workspace_size_ex (QMOE_ERR_INVALID_ARG / QMOE_ERR_UNSUPPORTED), and
 * QMOE_ERR_INVALID_ARG for a null info pointer or num_sms < 0.
 */
typedef struct {
  int32_t token_tile;
  int32_t issuers;
  int32_t acc_bufs;
  int32_t split1;
  int32_t split2;
  int32_t w_stages;
  int32_t ab_stages;
  int32_t stage_bytes;
  int64_t workspace_bytes;
  int32_t b_stages;
  int32_t dq_sets;
  int32_t cta_pair;
  int32_t cta_pair_down;
  int32_t reserved[2];
} qmoe_plan_info;

qmoe_status qmoe_describe_plan(const qmoe_layer* layer, int64_t M, int32_t top_k, const qmoe_options* opts,
                               int32_t num_sms, qmoe_plan_info* info);

/*
 * The fused MoE layer ("Marlin moe integration", description and review
 * thread: the hot-path call takes the activations, the already-quantized
 * expert weights and scales, and the router's top-k ids and weights, and runs
 * the grouped expert GEMMs; "[Kernel] W8A16 Int8 inside FusedMoE",
 * description: the int8 weights are cast to FP16/BF16 inside the kernel
 * before the matmul).
 * out[M, H] (act_dtype, overwritten) = the layer applied to x[M, H] (act_dtype)
 * with routing topk_ids int32 [M, top_k] and topk_weights float32 [M, top_k].
 * All buffers are device memory; x, out and the workspace 256-byte aligned.
 * workspace: at least qmoe_workspace_size bytes; its contents need no
 * initialisation and are scratch after the call.  Two forwards that share a
 * workspace must be ordered on the GPU (same stream or events).
 * Requirements: 1 <= top_k <= E; M*top_k < 2^31.  M == 0 launches nothing.
 */
qmoe_status qmoe_forward(const qmoe_layer* layer, const void* x, int64_t M,
                         const int32_t* topk_ids, const float* topk_weights, int32_t top_k,
                         void* out, void* workspace, size_t workspace_bytes, void* stream);
qmoe_status qmoe_forward_ex(const qmoe_layer* layer, const void* x, int64_t M,
                            const int32_t* topk_ids, const float* topk_weights, int32_t top_k,
                            void* out, void* workspace, size_t workspace_bytes, void* stream,
                            const qmoe_options* opts);

/*
 * qmoe_forward_ex with CUDA events recorded around each kernel launch, for
 * measuring per-kernel device time inside a timed region.  `events` holds
 * n_events (>= 14) cudaEvent_t handles created by the caller; for launch i
 * (0 moe_align, 1 token gather, 2 gate/up GEMM, 3 split-K SiLU reduce,
 * 4 intermediate rescale, 5 down GEMM, 6 output reduce) event 2i is recorded
 * on `stream` just before
 * it and event 2i+1 just after.  A launch the plan skips (3 when the gate/up
 * GEMM is not split; 1 for batches of at most 1024 token-expert pairs, whose
 * gather runs inside launch 0) gets both events at the same point.  *n_launches
 * (optional) receives the number of kernels launched.  Null events give
 * QMOE_ERR_INVALID_ARG.
 */
qmoe_status qmoe_forward_profiled(const qmoe_layer* layer, const void* x, int64_t M,
                                  const int32_t* topk_ids, const float* topk_weights, int32_t top_k,
                                  void* out, void* workspace, size_t workspace_bytes, void* stream,
                                  const qmoe_options* opts, void* const* events, int32_t n_events,
                                  int32_t* n_launches);

/*
 * Same layer with x, topk_ids, topk_weights and out in HOST memory; out is
 * valid once `stream` has been synchronised.  When all four are page-locked
 * buffers mapped into the device's address space (cudaHostAlloc memory on a
 * unified-addressing system, e.g. pinned memory on a Grace-Blackwell node,
 * where the GPU reaches it over NVLink-C2C) with x and out 256-byte aligned,
 * the forward's kernels read the inputs and write out in place and no copy is
 * enqueued.  Otherwise the call enqueues host-to-device copies of the inputs
 * into device staging, the forward, and the device-to-host copy of out
 * (page-locked memory makes those copies asynchronous).  The workspace
 * (device) must hold qmoe_workspace_size_host bytes (the staging lives in it).
 */
size_t qmoe_workspace_size_host(const qmoe_layer* layer, int64_t M, int32_t top_k);
qmoe_status qmoe_forward_host(const qmoe_layer* layer, const void* x_host, int64_t M,
                              const int32_t* topk_ids_host, const float* topk_weights_host, int32_t top_k,
                              void* out_host, void* workspace, size_t workspace_bytes, void* stream);

/*
 * qmoe_forward for callers that cannot allocate device memory at call time --
 * for example an inference-engine plugin whose memory plan is fixed before it
 * runs and that is handed no scratch buffer, or a serving loop that must not
 * enter an allocator (cudaMalloc can synchronise the device).  The pages have
 * no counterpart to this entry point.
 *
 * The forward's scratch is a 64 MiB array of device memory inside the library
 * image (resident on every GPU that loads the library until the process
 * exits); the call allocates nothing.  x, topk_ids, topk_weights and out are
 * as for qmoe_forward.  A layer/M/top_k whose qmoe_workspace_size exceeds
 * 64 MiB gives QMOE_ERR_WORKSPACE and launches nothing.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture on the device.
 *   - All calls share the one array, so calls whose GPU work overlaps (other
 *     streams, other host threads) race on it and give wrong results; order
 *     them on the GPU.  The array keeps the last call's contents; the forward
 *     needs none of it cleared.
 *   - Device-side faults (a bad expert id, a kernel wait timeout) are recorded
 *     in the shared array; qmoe_read_noalloc_status reads them back.
 *   - Invalid arguments give the same status as qmoe_forward, also at M == 0.
 */
qmoe_status qmoe_forward_noalloc(const qmoe_layer* layer, const void* x, int64_t M,
                                 const int32_t* topk_ids, const float* topk_weights, int32_t top_k,
                                 void* out, void* stream);

/*
 * Synchronise `stream` and return the first device-side fault recorded by the
 * most recent qmoe_forward_noalloc on the current device (QMOE_OK if none, or
 * if none has run).  Like that entry point it has no counterpart on the pages.
 */
qmoe_status qmoe_read_noalloc_status(void* stream);

/*
 * Router, the step before the layer (the pages take its output, the top-k
 * expert ids and weights, as the fused kernel's input; the Mixtral-style
 * layers they run route by softmax, top-k and renormalisation).  For each
 * token row of logits [M, E] (logits_dtype QMOE_F32, QMOE_F16 or QMOE_BF16,
 * device memory): topk_ids int32 [M, top_k] = the top_k experts by logit in
 * descending order, ties going to the lower expert id; topk_weights float32
 * [M, top_k] = their softmax probabilities exp(l_e) / sum_j exp(l_j),
 * divided by the sum of the kept ones when renormalize != 0.  NaN logits
 * count as -inf; a row of -inf logits routes uniformly.  Computed in fp32.
 * Requirements: 1 <= E <= 1024, 1 <= top_k <= E (QMOE_ERR_INVALID_ARG), and
 * top_k <= 32 (QMOE_ERR_UNSUPPORTED).  Asynchronous on `stream`.
 */
qmoe_status qmoe_route_topk(const void* logits, qmoe_dtype logits_dtype, int64_t M, int32_t E, int32_t top_k,
                            int32_t renormalize, int32_t* topk_ids, float* topk_weights, void* stream);

/*
 * The router then the layer in one call: out = the layer applied to x with
 * the routing qmoe_route_topk computes from logits (E = layer->E).  The
 * routing is kept in the workspace, which needs qmoe_workspace_size_logits
 * bytes (0 on invalid input); arguments otherwise as for qmoe_forward.
 */
size_t qmoe_workspace_size_logits(const qmoe_layer* layer, int64_t M, int32_t top_k);
qmoe_status qmoe_forward_logits(const qmoe_layer* layer, const void* x, int64_t M, const void* logits,
                                qmoe_dtype logits_dtype, int32_t top_k, int32_t renormalize, void* out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense linear layer                                                        */
/* ------------------------------------------------------------------------ */

/*
 * A dense linear layer out = x . W^T with W [N, K] weight-only quantized in
 * any of the formats above ("Add GPTQ Marlin 2:4 sparse structured support":
 * the GPTQ Marlin linear layer, 4 or 8 bits, group 128 or channel-wise, dense
 * or 2:4 sparse).  It runs the MoE layer's GEMM kernel with one weight matrix
 * and no routing or activation function.
 *   N, K         output and input features (multiples of 128).
 *   group_size, qt, act_dtype, scale_dtype   as for qmoe_layer.
 *   w            packed by qmoe_pack_linear (qmoe_packed_bytes(qt, 1, N, K,
 *                group_size) bytes), 256-byte aligned.
 *   s            per-column int8 and channel-wise 2:4-sparse int8: float32
 *                [N] (s_packed of qmoe_pack_linear); NULL otherwise.
 *   perm         int4 act-order (QMOE_INT4_GROUP / _ZP, group 128): int32 [K]
 *                written by qmoe_pack_linear; NULL otherwise.
 */
typedef struct {
  int32_t N, K;
  int32_t group_size;
  qmoe_quant_type qt;
  qmoe_dtype act_dtype;
  qmoe_dtype scale_dtype;
  const void* w;
  const float* s;
  const int32_t* perm;
} qmoe_linear;

/*
 * Pack one weight matrix for qmoe_linear (host memory in and out).
 *   q      codes [N, K], one per byte: uint8 0..15 (int4 formats) or int8
 *          -127..127 (int8 formats); 2:4 formats as for the MoE packers.
 *   s      scales: uint16 bit patterns of scale_dtype [K/128 (1 when
 *          group_size is -1), N] for the int4 formats, grouped int8 and
 *          grouped 2:4 int8; float [N] (scale_dtype QMOE_F32) for per-column
 *          int8 and channel-wise 2:4 int8.
 *   z      QMOE_INT4_GROUP_ZP only: zero points uint8 [K/128 or 1, N]; NULL otherwise.
 *   g_idx  int4 / int4 with zero points, group 128: int32 [K] act-order
 *          groups (each group exactly 128 channels) or NULL.
 * Outputs: w_packed (qmoe_packed_bytes(qt, 1, N, K, group_size) bytes);
 * s_packed float [N] for the float-scale formats (ignored otherwise);
 * perm_out int32 [K] when g_idx != NULL.  Errors as for the MoE packers.
 */
qmoe_status qmoe_pack_linear(qmoe_quant_type qt, int32_t N, int32_t K, int32_t group_size, qmoe_dtype scale_dtype,
                             const void* q, const void* s, const uint8_t* z, const int32_t* g_idx,
                             void* w_packed, float* s_packed, int32_t* perm_out);

/* Exact inverse of qmoe_pack_linear given the same g_idx (q, s, z as its inputs). */
qmoe_status qmoe_unpack_linear(qmoe_quant_type qt, int32_t N, int32_t K, int32_t group_size, const void* w_packed,
                               const float* s_packed, const int32_t* g_idx, void* q, void* s, uint8_t* z);

/* Workspace bytes of qmoe_linear_forward (0 on invalid input); opts may be NULL. */
size_t qmoe_linear_workspace_size(const qmoe_linear* layer, int64_t M, const qmoe_options* opts);

/* The launch plan of qmoe_linear_forward, as qmoe_describe_plan (split1 is its split-K, split2 0). */
qmoe_status qmoe_linear_describe_plan(const qmoe_linear* layer, int64_t M, const qmoe_options* opts,
                                      int32_t num_sms, qmoe_plan_info* info);

/*
 * out[M, N] (act_dtype, overwritten) = x[M, K] (act_dtype) . W^T, f16 MMA
 * operands with fp32 accumulation (as the MoE layer).  Device buffers; x, out
 * and the workspace 256-byte aligned; the workspace needs
 * qmoe_linear_workspace_size bytes.  opts: split1 (split-K), token_tile,
 * issuers, token_ring as for qmoe_forward_ex (NULL: automatic).  M == 0
 * launches nothing.  Asynchronous on `stream`; device-side faults are read
 * with qmoe_read_device_status on the workspace.
 */
qmoe_status qmoe_linear_forward(const qmoe_linear* layer, const void* x, int64_t M, void* out,
                                void* workspace, size_t workspace_bytes, void* stream,
                                const qmoe_options* opts);

/*
 * Synchronise `stream` and return the first device-side fault recorded in
 * `workspace` by the most recent forward that used it (QMOE_OK if none).
 */
qmoe_status qmoe_read_device_status(const void* workspace, void* stream);

/* Static description of a status code. */
const char* qmoe_status_string(qmoe_status status);

/* QMOE_ABI_VERSION of the loaded library. */
int32_t qmoe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H_ */
