// api.cpp - host side of libqmoe: argument validation, weight packing,
// workspace planning and the launch sequence of the fused MoE forward.  The C
// ABI is declared in include/qmoe.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "qmoe.h"
#include "qmoe_internal.h"

namespace qmoe {
namespace {

constexpr size_t kMaxDynSmem = 232448;  // 227 KB per CTA on sm_100-class GPUs
constexpr int kDefaultSms = 152;

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// small host utilities
// ---------------------------------------------------------------------------
template <class F>
void parallel_for(int64_t n, F&& f) {
  const int64_t hw = std::max<int64_t>(1, std::thread::hardware_concurrency());
  const int64_t nt = std::min<int64_t>(hw, n);
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> ts;
  for (int64_t t = 0; t < nt; ++t)
    ts.emplace_back([&] {
      for (int64_t i = next++; i < n; i = next++) f(i);
    });
  for (auto& t : ts) t.join();
}

int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return kDefaultSms;
  }
  static std::mutex mu;
  static int cache[128] = {0};
  std::lock_guard<std::mutex> lk(mu);
  if (dev >= 0 && dev < 128 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return kDefaultSms;
  }
  if (dev >= 0 && dev < 128) cache[dev] = n;
  return n;
}

qmoe_status check_dev_ptr(const void* p, int dev) {
  if (p == nullptr) return QMOE_ERR_INVALID_ARG;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_DEVICE_MISMATCH;
  }
  if (a.type == cudaMemoryTypeManaged) return QMOE_OK;
  if (a.type != cudaMemoryTypeDevice || a.device != dev) return QMOE_ERR_DEVICE_MISMATCH;
  return QMOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of a page-locked host buffer mapped into the device's address
// space, else nullptr (pageable or device memory, or an unknown pointer).
const void* mapped_host_ptr(const void* p) {
  if (p == nullptr) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// ---------------------------------------------------------------------------
// layer validation and the forward plan
// ---------------------------------------------------------------------------
int stage_bytes_of(int32_t qt, int32_t gs) {
  switch (qt) {
    case QMOE_INT4_GROUP: return kInt4StageBytes;
    case QMOE_INT4_GROUP_ZP: return kInt4ZpStageBytes;
    case QMOE_INT8_GROUP: return kInt8GroupStageBytes;
    case QMOE_INT4_GROUP_24: return kInt4SparseStageBytes;
    case QMOE_INT8_24: return gs == -1 ? kInt8SparseStageBytes : kInt8SparseGroupStageBytes;
    default: return kInt8StageBytes;
  }
}

QuantKind kind_of(int32_t qt, int32_t gs) {
  switch (qt) {
    case QMOE_INT4_GROUP: return kQ4;
    case QMOE_INT4_GROUP_ZP: return kQ4Z;
    case QMOE_INT8_GROUP: return kQ8G;
    case QMOE_INT4_GROUP_24: return kQ4S;
    case QMOE_INT8_24: return gs == -1 ? kQ8S : kQ8SG;
    default: return kQ8;
  }
}

// Formats whose scales are one float32 per output feature, outside the packed blocks
// (applied to the accumulator in the GEMM epilogue).
bool has_row_scales(int32_t qt, int32_t gs) {
  return qt == QMOE_INT8_PER_COL || (qt == QMOE_INT8_24 && gs == -1);
}

// Format, group size, scale type and act-order checks shared by the MoE layer
// and the dense linear layer.
qmoe_status validate_format(int32_t qt, int32_t gs, int32_t act, int32_t sdt, bool has_perm) {
  if (act != QMOE_F16 && act != QMOE_BF16) return QMOE_ERR_UNSUPPORTED;
  if (qt == QMOE_INT4_GROUP || qt == QMOE_INT4_GROUP_ZP) {
    if (gs != 128 && gs != -1) return QMOE_ERR_UNSUPPORTED;
    if (sdt != act) return QMOE_ERR_UNSUPPORTED;
    if (gs == -1 && has_perm) return QMOE_ERR_UNSUPPORTED;
  } else if (qt == QMOE_INT4_GROUP_24) {
    if (gs != 128 && gs != -1) return QMOE_ERR_UNSUPPORTED;
    if (sdt != act) return QMOE_ERR_UNSUPPORTED;
    if (has_perm) return QMOE_ERR_UNSUPPORTED;
  } else if (qt == QMOE_INT8_GROUP) {
    if (gs != 128) return QMOE_ERR_UNSUPPORTED;
    if (sdt != act) return QMOE_ERR_UNSUPPORTED;
    if (has_perm) return QMOE_ERR_UNSUPPORTED;
  } else if (qt == QMOE_INT8_PER_COL) {
    if (gs != -1) return QMOE_ERR_UNSUPPORTED;
    if (sdt != QMOE_F32) return QMOE_ERR_UNSUPPORTED;
    if (has_perm) return QMOE_ERR_UNSUPPORTED;
  } else if (qt == QMOE_INT8_24) {
    if (gs != 128 && gs != -1) return QMOE_ERR_UNSUPPORTED;
    if (sdt != (gs == -1 ? QMOE_F32 : act)) return QMOE_ERR_UNSUPPORTED;
    if (has_perm) return QMOE_ERR_UNSUPPORTED;
  } else {
    return QMOE_ERR_INVALID_ARG;
  }
  return QMOE_OK;
}

// Act-order gathers stage one token row (2 bytes per channel) in shared memory.
constexpr int32_t kMaxActOrderK = 65536;

qmoe_status validate_layer_dims(const qmoe_layer* L) {
  if (L == nullptr) return QMOE_ERR_INVALID_ARG;
  if (L->E < 1 || L->E > 1024 || L->H <= 0 || L->I <= 0) return QMOE_ERR_INVALID_ARG;
  if (L->H % 128 != 0 || L->I % 128 != 0) return QMOE_ERR_UNSUPPORTED;
  if (L->perm13 != nullptr && L->H > kMaxActOrderK) return QMOE_ERR_UNSUPPORTED;
  return validate_format(L->qt, L->group_size, L->act_dtype, L->scale_dtype, L->perm13 != nullptr);
}

struct Plan {
  int64_t M = 0, P = 0;
  int k = 0;
  int T = 0, acc_bufs = 0, issuers = 0, a_col0 = 0, stage_bytes = 0, w_stages = 0, ab_stages = 0, b_stages = 0;
  int dq_sets = 2;
  int pg = 0, d_col0 = 0;
  int S1 = 1, S2 = 1;
  int n_tiles1 = 0, n_tiles2 = 0, kst1 = 0, kst2 = 0;
  int64_t cap = 0, nblocks = 0, max_chunks = 0;
  size_t off_status = 0, off_sorted = 0, off_expert = 0, off_scalars = 0, off_chunks = 0, off_xg = 0, off_xscale = 0,
         off_inter32 = 0, off_inter16 = 0, off_iscale = 0, off_h = 0, off_y = 0, off_c13 = 0, off_c2 = 0, total = 0;
  int fused_reduce = 0;  // top-k reduction in the down GEMM's epilogue
  size_t off_cnt = 0;
  int pair = 0;          // GEMMs on CTA pairs (M = 256 MMAs, half the token rows per CTA)
  // the down GEMM's launch shape where it differs from the gate/up GEMM's
  struct Rings {
    int issuers = 0, acc_bufs = 0, a_col0 = 0, w_stages = 0, ab_stages = 0, b_stages = 0, dq_sets = 2, pair = 0;
  } r2;
};

Plan::Rings rings_of(const Plan& p) {
  Plan::Rings r;
  r.issuers = p.issuers;
  r.acc_bufs = p.acc_bufs;
  r.a_col0 = p.a_col0;
  r.w_stages = p.w_stages;
  r.ab_stages = p.ab_stages;
  r.b_stages = p.b_stages;
  r.dq_sets = p.dq_sets;
  r.pair = p.pair;
  return r;
}

// Makespan, in pipeline stages, of n work items of k stages each split s ways
// over C persistent CTAs.  A CTA's items run back to back; each item costs the
// longer of its stages and its epilogue (`epi` stages' worth, overlapped with
// the next item's stages when TMEM holds two accumulator buffers).  Each split
// beyond the first adds `reduce` stages' worth of partial-sum traffic.
double split_cost(int64_t n, int k, int s, int C, double epi, double reduce) {
  const int64_t per_cta = (n * s + C - 1) / C;
  return static_cast<double>(per_cta) * std::max(static_cast<double>(k) / s, epi) + reduce * (s - 1);
}

int choose_split(int64_t n_items, int k_stages, int C, double epi, double reduce, double must_gain) {
  const int smax = std::max(1, std::min(64, k_stages / 4));
  int best = 1;
  double best_cost = split_cost(n_items, k_stages, 1, C, epi, reduce);
  const double base = best_cost;
  for (int s = 2; s <= smax; ++s) {
    const double c = split_cost(n_items, k_stages, s, C, epi, reduce);
    if (c < best_cost) {
      best_cost = c;
      best = s;
    }
  }
  return best_cost < base * must_gain ? best : 1;
}

// Work-item raster of a GEMM (GemmParams::chunk_group, see decode_item): with
// two or more chunks per expert on average, groups follow the experts, each at
// most as many chunks as keep its token tiles (T rows x K x 2 bytes each) within
// 32 MB, a quarter of L2, so each weight tile is read from HBM once per group;
// otherwise groups of 8 consecutive chunks (several experts' tiles side by
// side).  Measured on GB300 (Mixtral-8x22B shape, DRAM bytes per launch): at
// M = 2048 gate/up 1.55 -> 1.13 GB and down 1.07 -> 0.69 GB against fixed
// groups of 8 chunks; a 64 MB budget made the M = 8192 down GEMM's 16-chunk
// groups re-read their token tiles (2.9 -> 3.7 GB).
int chunk_raster(int64_t P, int E, int T, int64_t K) {
  if (P < 2LL * E * T) return 8;
  const int64_t per_chunk = static_cast<int64_t>(T) * K * 2;
  return -static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(1 << 20, (int64_t(32) << 20) / per_chunk)));
}

// Issuers, TMEM accumulators and ring depths of the GEMM for the token tile
// p->T and the packed block size p->stage_bytes (shared by the MoE layer and the
// dense linear layer).
qmoe_status size_gemm_rings(const qmoe_options* o, Plan* p) {
  // MMA issuers (stage g to issuer g mod n, one accumulator each): with small
  // token tiles one issuing warp's rate, with the wait and commit around each
  // stage, is below what the tensor core accepts, so tiles up to 64 rows take
  // two; a 128-row tile keeps the tensor pipe busy from one warp, which leaves
  // TMEM for two accumulator buffers so the epilogue overlaps the next item's
  // MMAs.  (Measured on GB300: two issuers 1-5 % faster than three and 5-16 %
  // faster than one at 16-64 rows for every weight format; one issuer 9 %
  // faster than two at 128 rows, Mixtral-8x7B int4 M = 256.)
  const int T = p->T;
  p->issuers = (T <= 64) ? 2 : 1;
  if (o != nullptr && o->issuers != 0) {
    if (o->issuers < 1 || o->issuers > 3) return QMOE_ERR_INVALID_ARG;
    p->issuers = o->issuers;
  }
  // Ring sizes are multiples of every role's stride (2 for the producers and
  // dequant sets, the issuer count for the issuers): each slot then belongs to
  // one role of each kind, and each waiter sees every phase of its barriers.
  // (Otherwise a role would see only some uses of a slot and a parity wait
  // could pass on a phase two behind.)
  const int ring_mult = (p->issuers == 3) ? 6 : 2;
  // TMEM (512 columns): accumulators (issuers x buffers x T columns), then the
  // 64-column A slots paired with the token-tile ring (at most 8)
  auto a_slots = [&](int accb) {
    const int n = std::min(8, (512 - p->issuers * accb * T) / 64);
    return n / ring_mult * ring_mult;
  };
  if (p->pg) {
    // per-group scaling: no accumulators; each A slot has a 16-column D slot after the A slots
    p->acc_bufs = 1;
    p->a_col0 = 0;
    p->ab_stages = std::min(8, 512 / (64 + 16)) / ring_mult * ring_mult;
    p->d_col0 = 64 * p->ab_stages;
  } else {
    p->acc_bufs = a_slots(2) >= ring_mult ? 2 : 1;
    p->a_col0 = p->issuers * p->acc_bufs * T;
    p->ab_stages = a_slots(p->acc_bufs);
  }
  if (p->ab_stages < ring_mult) return (o != nullptr && o->issuers != 0) ? QMOE_ERR_INVALID_ARG : QMOE_ERR_UNSUPPORTED;
  // Token-tile ring: a multiple m of the A ring, so that a token tile can be
  // fetched up to m - 1 A-ring laps before its MMAs and its L2 latency stays
  // off the A slots' cycle.  The deepest m <= 2 that leaves the weight ring at
  // least 8 slots (weights stream from HBM and want the deeper ring).
  const size_t wslot = (static_cast<size_t>(p->stage_bytes) + 1023) & ~size_t(1023);
  auto w_depth = [&](int nb2) {
    // (+ the per-group-scaled int4 epilogue's staging buffers)
    // (a CTA of a pair holds half of each token tile's rows)
    const size_t b_bytes = static_cast<size_t>(nb2) * T * (p->pair ? 128 : 256) + (p->pg ? kPgStageBytes : 0);
    if (b_bytes + 2048 + 2 * wslot > kMaxDynSmem) return 0;
    return static_cast<int>(std::min<size_t>(16, (kMaxDynSmem - 2048 - b_bytes) / wslot)) & ~1;
  };
  // large token tiles: fewer A slots (hence token-tile slots) where shared memory
  // would otherwise hold too few weight slots
  while (p->ab_stages > ring_mult && w_depth(p->ab_stages) < 4) p->ab_stages -= ring_mult;
  int ring_m = 1;
  if (o != nullptr && o->token_ring != 0) {
    if (o->token_ring < 1 || o->token_ring > 3) return QMOE_ERR_INVALID_ARG;
    ring_m = o->token_ring;
    if (w_depth(ring_m * p->ab_stages) < 2) return QMOE_ERR_INVALID_ARG;
  } else {
    for (int m = 2; m > 1; --m)
      if (w_depth(m * p->ab_stages) >= 8) {
        ring_m = m;
        break;
      }
  }
  p->b_stages = ring_m * p->ab_stages;
  p->w_stages = w_depth(p->b_stages);
  if (p->w_stages < 2 || p->ab_stages < 2) return QMOE_ERR_UNSUPPORTED;
  // Dequant sets: 4 sets of 4 warps (each converts whole stage rows for its 32
  // rows) or 2 sets of 8 warps (each converts half rows).  A set takes every
  // DS-th stage, so the weight ring and the token-tile ring must be multiples of
  // DS for each slot's barriers to belong to one set.  Four sets halve the
  // per-stage wait / store / arrive work of the dequant warps and keep four
  // stages in conversion at once (measured on GB300: 3-10 % faster at every
  // size, most at decode), so they are chosen wherever the rings allow.
  if (o != nullptr && (o->weight_l2 < 0 || o->weight_l2 > 2)) return QMOE_ERR_INVALID_ARG;
  // (a set starts at A slot `set` and steps by the set count: at least 4 A slots)
  const bool four_ok = (p->w_stages & ~3) >= 4 && p->b_stages % 4 == 0 && p->ab_stages >= 4;
  p->dq_sets = four_ok ? 4 : 2;
  if (o != nullptr && o->dq_sets != 0) {
    if (o->dq_sets != 2 && o->dq_sets != 4) return QMOE_ERR_INVALID_ARG;
    if (o->dq_sets == 4 && !four_ok) return QMOE_ERR_INVALID_ARG;
    p->dq_sets = o->dq_sets;
  }
  if (p->dq_sets == 4) p->w_stages &= ~3;
  return QMOE_OK;
}

qmoe_status make_plan(const qmoe_layer* L, int64_t M, int32_t k, const qmoe_options* o, int sms, Plan* pl) {
  qmoe_status st = validate_layer_dims(L);
  if (st != QMOE_OK) return st;
  if (M < 0 || k < 1 || k > L->E) return QMOE_ERR_INVALID_ARG;
  if (M * static_cast<int64_t>(k) >= (int64_t(1) << 31) - int64_t(L->E) * kAlignBlock) return QMOE_ERR_UNSUPPORTED;
  Plan p;
  p.M = M;
  p.k = k;
  p.P = M * k;
  const int64_t P = p.P;
  // token tile: a power of two from 16 to 128, at least 1.5 times the mean
  // number of pairs per expert, so that each expert's rows are usually one chunk
  // (measured on GB300: Mixtral M = 16 -> 16 rows, 64 -> 32, 128 -> 64, 256 ->
  // 128; 160 experts top-6 at M = 1024 -> 64)
  int T = 16;
  while (T < 128 && 2 * T * static_cast<int64_t>(L->E) < 3 * P) T *= 2;
  // A token adds at most one pair to an expert, so an expert's rows can reach M,
  // E/k times the mean.  Where that ratio is large (fine-grained experts) an
  // uneven router sends several 16-row chunks to its busiest experts, each
  // dequantizing the same weights again: plan at least 32 rows there once M
  // can fill them.  (Measured on GB300 with 160 experts top-6: under a
  // Zipf(1.1)-biased router 3-17 % faster at M = 32..256; under an unbiased
  // one at most 0.9 % slower.)
  if (T < 32 && L->E >= 16 * k && M >= 32) T = 32;
  if (o != nullptr && o->token_tile != 0) {
    if (o->token_tile < 16 || o->token_tile > kMaxTokenTile || o->token_tile % 16 != 0) return QMOE_ERR_INVALID_ARG;
    T = o->token_tile;
  }
  p.T = T;
  p.stage_bytes = stage_bytes_of(L->qt, L->group_size);
  // Per-group scaling (symmetric int4, 16-row token tiles): the dequant warps keep
  // only the magic-number unpacks and the epilogue warps apply each group's scale
  // in fp32 (the scale multiply and zero-point subtract were ~12 % of the int4
  // decode GEMM's time in an ablation on GB300).
  if (o != nullptr && (o->int4_group_epilogue < 0 || o->int4_group_epilogue > 2)) return QMOE_ERR_INVALID_ARG;
  // Automatic: off (measured on GB300 with Mixtral-8x7B int4 at M = 16: the four
  // epilogue warps need ~1000 cycles per stage, above the standard path's ~650).
  const bool pg_ok = L->qt == QMOE_INT4_GROUP && T == 16;
  if (o != nullptr && o->int4_group_epilogue == 1 && !pg_ok) return QMOE_ERR_INVALID_ARG;
  p.pg = (pg_ok && o != nullptr && o->int4_group_epilogue == 1) ? 1 : 0;
  // CTA pairs (option cta_pair: 0 automatic, 1 on, 2 off): symmetric int4 and
  // per-channel int8 with the standard epilogues
  if (o != nullptr && (o->cta_pair < 0 || o->cta_pair > 2)) return QMOE_ERR_INVALID_ARG;
  const bool pair_ok = (L->qt == QMOE_INT4_GROUP || L->qt == QMOE_INT8_PER_COL) && !p.pg &&
                       !(o != nullptr && o->topk_reduce == 1);
  if (o != nullptr && o->cta_pair == 1 && !pair_ok) return QMOE_ERR_INVALID_ARG;
  p.pair = (o != nullptr && o->cta_pair == 1) ? 1 : 0;
  p.n_tiles1 = 2 * L->I / kTileRows;
  p.n_tiles2 = L->H / kTileRows;
  p.kst1 = L->H / kStageK;
  p.kst2 = L->I / kStageK;
  if ((st = size_gemm_rings(o, &p)) != QMOE_OK) return st;
  // Automatic CTA pairs where shared memory held the single-CTA rings short (a
  // token-tile ring of one A-ring depth, or fewer than 8 weight slots): each CTA
  // of a pair holds half of every token tile, so the pair gets the deeper rings
  // (measured on GB300: Mixtral-8x22B int4 prefill 7-10 % faster, Mixtral-8x7B
  // int4 M = 512 8 %, int8 M = 128 and 512 9 % and 3 %, 160 experts top-6 int8
  // M = 1024 7.5 %; where the rings were already deep, pairs were ~2 % slower).
  if (pair_ok && (o == nullptr || (o->cta_pair == 0 && o->token_ring == 0)) &&
      (p.b_stages == p.ab_stages || p.w_stages < 8)) {
    p.pair = 1;
    if ((st = size_gemm_rings(o, &p)) != QMOE_OK) return st;
  }
  // The down GEMM on single CTAs where its K spans fewer than 32 stages: its
  // items are then too short for the pair's deeper rings to pay for the pair's
  // per-item fill and epilogue (measured on GB300 with 160 experts top-6, K =
  // 1536 in 12 stages: 4 % slower on pairs at M = 1024, while every down GEMM
  // with K of 112-128 stages was 2-13 % faster).
  p.r2 = rings_of(p);
  if (p.pair && (o == nullptr || o->cta_pair == 0) && p.kst2 < 32) {
    Plan q = p;
    q.pair = 0;
    if (size_gemm_rings(o, &q) == QMOE_OK) p.r2 = rings_of(q);
  }
  // rows of the staged B operands: a multiple of 16 (whole 8-row swizzle groups)
  p.cap = (P + static_cast<int64_t>(L->E) * (kAlignBlock - 1) + 15) / 16 * 16;
  p.nblocks = (p.cap + kAlignBlock - 1) / kAlignBlock;
  p.max_chunks = (p.cap + T - 1) / T + L->E;
  // expected chunks for the split heuristic (uniform routing)
  const double d = L->E * (1.0 - std::pow(1.0 - 1.0 / L->E, static_cast<double>(P)));
  const int64_t est_chunks = std::max<int64_t>(std::max<int64_t>(1, static_cast<int64_t>(std::ceil(d))), (P + T - 1) / T);
  // Epilogue time of one item in pipeline stages (measured on GB300: about 3k
  // cycles for a 16-row chunk, 15k for a 128-row one, against 0.7k-1.1k per
  // stage).  Partial sums of one extra split: written and read once in fp32,
  // in stage-times of the whole GPU's weight stream (~1.3 MB per stage-time),
  // plus two stages per split for the extra items' pipeline fill and drain
  // and for summing the partials (fitted on GB300: Mixtral-8x7B decode runs
  // its down GEMM fastest split 4 ways, not 7).
  const double epi = 4.0 + T / 8.0;
  const double stage_bytes_gpu = 1.3e6;
  p.S1 = choose_split(est_chunks * p.n_tiles1, p.kst1, sms, epi, 2.0 + 8.0 * P * 2 * L->I / stage_bytes_gpu, 0.8);
  p.S2 = choose_split(est_chunks * p.n_tiles2, p.kst2, sms, epi, 2.0 + 8.0 * P * L->H / stage_bytes_gpu, 0.99);
  if (o != nullptr && o->split1 != 0) {
    if (o->split1 < 1 || o->split1 > 64 || o->split1 > p.kst1) return QMOE_ERR_INVALID_ARG;
    p.S1 = o->split1;
  }
  if (o != nullptr && o->split2 != 0) {
    if (o->split2 < 1 || o->split2 > 64 || o->split2 > p.kst2) return QMOE_ERR_INVALID_ARG;
    p.S2 = o->split2;
  }

  // Top-k reduction: automatic = the separate kernel.  In the down GEMM's
  // epilogue (option 1) it saves a launch but was slower at every batch size
  // measured on GB300 (Mixtral-8x7B int4 M = 16: down GEMM 72 -> 115 us): the
  // last warp to arrive sums its tokens' partials with dependent L2 loads on
  // the epilogue's path.
  if (o != nullptr && (o->topk_reduce < 0 || o->topk_reduce > 2)) return QMOE_ERR_INVALID_ARG;
  p.fused_reduce = (o != nullptr && o->topk_reduce == 1) ? 1 : 0;

  size_t off = 0;
  p.off_status = off;   off += 256;
  p.off_sorted = off;   off += al256(p.cap * 4);
  p.off_expert = off;   off += al256(p.nblocks * 4);
  p.off_scalars = off;  off += 256;  // num_post_padded, n_chunks
  p.off_chunks = off;   off += al256(p.max_chunks * sizeof(Chunk));
  p.off_xg = off;       off += al256(static_cast<size_t>(p.cap) * L->H * 2);
  p.off_xscale = off;   off += al256(static_cast<size_t>(p.cap) * 4);
  p.off_inter32 = off;  off += al256(static_cast<size_t>(p.cap) * L->I * 4);
  p.off_inter16 = off;  off += al256(static_cast<size_t>(p.cap) * L->I * 2);
  p.off_iscale = off;   off += al256(static_cast<size_t>(p.cap) * 4);
  p.off_h = off;        off += (p.S1 > 1) ? al256(static_cast<size_t>(p.S1) * p.cap * 2 * L->I * 4) : 0;
  p.off_y = off;        off += al256(static_cast<size_t>(p.S2) * P * L->H * 4);
  if (p.fused_reduce) {
    p.off_cnt = off;    off += al256(static_cast<size_t>(M) * p.n_tiles2 * 4 * 4);
  }
  if (p.pg) {
    p.off_c13 = off;    off += al256(static_cast<size_t>(p.cap) * p.kst1 * 4);
    p.off_c2 = off;     off += al256(static_cast<size_t>(p.cap) * p.kst2 * 4);
  }
  p.total = off;
  *pl = p;
  return QMOE_OK;
}

// host_io: x, topk_ids, topk_weights and out are the device addresses of
// page-locked, device-mapped host buffers (checked by the caller); the kernels
// read and write them in place with plain loads and stores.
qmoe_status forward_impl(const qmoe_layer* L, const void* x, int64_t M, const int32_t* topk_ids,
                         const float* topk_weights, int32_t k, void* out, void* ws, size_t ws_bytes,
                         cudaStream_t stream, const qmoe_options* opts, void* const* events = nullptr,
                         int32_t* n_launches = nullptr, bool host_io = false) {
  const int sms = current_sm_count();
  Plan pl;
  qmoe_status st = make_plan(L, M, k, opts, sms, &pl);
  if (st != QMOE_OK) return st;
  if (M == 0) return QMOE_OK;
  if (ws == nullptr || ws_bytes < pl.total) return QMOE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  const void* ptrs[] = {ws, L->w13, L->w2, x, topk_ids, topk_weights, out};
  const int n_checked = host_io ? 3 : 7;  // (host_io: the caller checked the four I/O buffers)
  for (int i = 0; i < n_checked; ++i)
    if ((st = check_dev_ptr(ptrs[i], dev)) != QMOE_OK) return st;
  // only per-column int8 keeps its scales outside the packed weight blocks
  const bool row_scales = has_row_scales(L->qt, L->group_size);
  if (row_scales) {
    if ((st = check_dev_ptr(L->s13, dev)) != QMOE_OK) return st;
    if ((st = check_dev_ptr(L->s2, dev)) != QMOE_OK) return st;
  }
  if (L->perm13 != nullptr && (st = check_dev_ptr(L->perm13, dev)) != QMOE_OK) return st;
  if (!aligned(x, 256) || !aligned(out, 256) || !aligned(ws, 256) || !aligned(L->w13, 256) ||
      !aligned(L->w2, 256) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
      (L->perm13 != nullptr && !aligned(L->perm13, 16)) ||
      (row_scales && (!aligned(L->s13, 16) || !aligned(L->s2, 16))))
    return QMOE_ERR_INVALID_ARG;

  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(base + pl.off_status);
  int32_t* sorted = reinterpret_cast<int32_t*>(base + pl.off_sorted);
  int32_t* expert = reinterpret_cast<int32_t*>(base + pl.off_expert);
  int32_t* npp = reinterpret_cast<int32_t*>(base + pl.off_scalars);
  int32_t* nch = npp + 1;
  Chunk* chunks = reinterpret_cast<Chunk*>(base + pl.off_chunks);
  void* xg = base + pl.off_xg;
  float* xscale = reinterpret_cast<float*>(base + pl.off_xscale);
  float* inter32 = reinterpret_cast<float*>(base + pl.off_inter32);
  void* inter16 = base + pl.off_inter16;
  float* iscale = reinterpret_cast<float*>(base + pl.off_iscale);
  float* h = reinterpret_cast<float*>(base + pl.off_h);
  float* y = reinterpret_cast<float*>(base + pl.off_y);
  // per-group corrections of the token operands (per-group-scaled int4 GEMM)
  float* c13 = pl.pg ? reinterpret_cast<float*>(base + pl.off_c13) : nullptr;
  float* c2 = pl.pg ? reinterpret_cast<float*>(base + pl.off_c2) : nullptr;
  const bool bf16 = L->act_dtype == QMOE_BF16;
  const int P = static_cast<int>(pl.P);


  // events (profiling only): 2i before and 2i+1 after launch i
  auto rec = [&](int idx) {
    if (events != nullptr) cudaEventRecord(static_cast<cudaEvent_t>(events[idx]), stream);
  };
  int launched = 0;
  cudaError_t err;
  if (align_gather_small_fits(P, L->E, kAlignBlock, L->H, L->perm13 != nullptr)) {
    // small batch: grouping and gather in one kernel (launch 1 then takes no time)
    rec(0);
    err = launch_align_gather_small(topk_ids, P, L->E, kAlignBlock, pl.cap, sorted, expert, npp, pl.T, chunks, nch,
                                    status, x, bf16, L->perm13, k, L->H, pl.cap, xg, xscale, c13, sms, stream);
    rec(1);
    launched += (err == cudaSuccess);
    rec(2);
    rec(3);
  } else {
    rec(0);
    err = launch_align(topk_ids, P, L->E, kAlignBlock, pl.cap, sorted, expert, npp, pl.T, chunks, nch, status, stream);
    rec(1);
    launched += (err == cudaSuccess);
    rec(2);
    if (err == cudaSuccess) {
      err = launch_gather(x, bf16, sorted, expert, npp, L->perm13, P, k, L->H, kAlignBlock, pl.cap, xg, xscale, c13,
                          sms, stream);
      launched += (err == cudaSuccess);
    }
    rec(3);
  }
  GemmParams g1{};
  g1.w = static_cast<const uint8_t*>(L->w13);
  g1.b = static_cast<const uint8_t*>(xg);
  g1.b_unit_stride = pl.cap * 256;
  g1.row_scale = row_scales ? L->s13 : nullptr;
  g1.col_scale = xscale;
  g1.chunks = chunks;
  g1.n_chunks = nch;
  g1.sorted_ids = sorted;
  g1.topk_w = topk_weights;
  g1.status = status;
  g1.n_tiles = pl.n_tiles1;
  g1.k_groups = pl.kst1;
  g1.split = pl.S1;
  g1.token_tile = pl.T;
  g1.acc_bufs = pl.acc_bufs;
  g1.a_col0 = pl.a_col0;
  g1.issuers = pl.issuers;
  g1.w_stages = pl.w_stages;
  g1.ab_stages = pl.ab_stages;
  g1.b_stages = pl.b_stages;
  g1.dq_sets = pl.dq_sets;
  g1.pg = pl.pg;
  g1.pair = pl.pair;
  g1.d_col0 = pl.d_col0;
  g1.pg_corr = c13;
  g1.pg_cap = pl.cap;
  g1.fault_injection = (opts != nullptr) ? opts->fault_injection : 0;
  g1.stage_bytes = pl.stage_bytes;
  g1.P = P;
  g1.chunk_group = chunk_raster(P, L->E, pl.T, L->H);
  g1.inter_ld = L->I;
  // more pairs per expert than a token tile holds: several chunks read each weight tile
  g1.w_shared = (opts != nullptr && opts->weight_l2 != 0) ? (opts->weight_l2 == 1)
                                                           : (pl.P > static_cast<int64_t>(L->E) * pl.T);
  if (pl.S1 == 1) {
    g1.epi_mode = kEpiSiluToAct;
    g1.out = inter32;
    g1.out_ld = L->I;
    g1.out_split_stride = 0;
  } else {
    g1.epi_mode = kEpiPartialRows;
    g1.out = h;
    g1.out_ld = 2LL * L->I;
    g1.out_split_stride = pl.cap * 2LL * L->I;
  }
  GemmParams g2 = g1;
  g2.issuers = pl.r2.issuers;
  g2.acc_bufs = pl.r2.acc_bufs;
  g2.a_col0 = pl.r2.a_col0;
  g2.w_stages = pl.r2.w_stages;
  g2.ab_stages = pl.r2.ab_stages;
  g2.b_stages = pl.r2.b_stages;
  g2.dq_sets = pl.r2.dq_sets;
  g2.pair = pl.r2.pair;
  g2.w = static_cast<const uint8_t*>(L->w2);
  g2.b = static_cast<const uint8_t*>(inter16);
  g2.b_unit_stride = pl.cap * 256;
  g2.row_scale = row_scales ? L->s2 : nullptr;
  g2.col_scale = iscale;
  g2.n_tiles = pl.n_tiles2;
  g2.k_groups = pl.kst2;
  g2.chunk_group = chunk_raster(P, L->E, pl.T, L->I);
  g2.split = pl.S2;
  g2.epi_mode = kEpiWeightedPairs;
  g2.pg_corr = c2;
  g2.fault_injection = 0;
  g2.out = y;
  g2.out_ld = L->H;
  g2.out_split_stride = pl.P * static_cast<int64_t>(L->H);
  if (pl.fused_reduce) {
    g2.red_cnt = reinterpret_cast<int32_t*>(base + pl.off_cnt);
    g2.topk_ids = topk_ids;
    g2.red_out = static_cast<uint16_t*>(out);
    g2.top_k = k;
    g2.n_experts = L->E;
    g2.out_bf16 = bf16 ? 1 : 0;
  }

  // (CTA pairs: work items over tile pairs, two CTAs per item)
  const int64_t items1 = pl.max_chunks * (pl.pair ? (pl.n_tiles1 + 1) / 2 : pl.n_tiles1) * pl.S1;
  const int64_t items2 = pl.max_chunks * (pl.r2.pair ? (pl.n_tiles2 + 1) / 2 : pl.n_tiles2) * pl.S2;
  const int grid1 = pl.pair ? 2 * static_cast<int>(std::min<int64_t>(sms / 2, items1))
                            : static_cast<int>(std::min<int64_t>(sms, items1));
  const int grid2 = pl.r2.pair ? 2 * static_cast<int>(std::min<int64_t>(sms / 2, items2))
                            : static_cast<int>(std::min<int64_t>(sms, items2));
  rec(4);
  if (err == cudaSuccess) {
    err = launch_gemm(kind_of(L->qt, L->group_size), bf16, g1, grid1, stream);  // in-block scales have the activation dtype
    launched += (err == cudaSuccess);
  }
  rec(5);
  rec(6);
  if (err == cudaSuccess && pl.S1 > 1) {
    err = launch_silu_reduce(h, npp, pl.S1, pl.cap, L->I, inter32, sms, stream);
    launched += (err == cudaSuccess);
  }
  rec(7);
  rec(8);
  if (err == cudaSuccess) {
    TopkPrep prep{};
    if (pl.fused_reduce) {
      prep.cnt = g2.red_cnt;
      prep.n_cnt = M * static_cast<int64_t>(pl.n_tiles2) * 4;
      prep.topk_ids = topk_ids;
      prep.M = M;
      prep.top_k = k;
      prep.E = L->E;
      prep.H = L->H;
      prep.out = static_cast<uint16_t*>(out);
    }
    err = launch_inter_rescale(inter32, npp, sorted, P, L->I, pl.cap, inter16, iscale, c2, prep, sms, stream);
    launched += (err == cudaSuccess);
  }
  rec(9);
  rec(10);
  if (err == cudaSuccess) {
    err = launch_gemm(kind_of(L->qt, L->group_size), bf16, g2, grid2, stream);
    launched += (err == cudaSuccess);
  }
  rec(11);
  rec(12);
  if (err == cudaSuccess && !pl.fused_reduce) {
    err = launch_out_reduce(y, topk_ids, L->E, pl.S2, M, k, L->H, bf16, out, sms, stream);
    launched += (err == cudaSuccess);
  }
  rec(13);
  if (n_launches != nullptr) *n_launches = launched;
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// dense linear layer: out[M, N] = x[M, K] . W^T with W [N, K] weight-only
// quantized in any of the packed formats (one GEMM, no routing, no SiLU)
// ---------------------------------------------------------------------------
struct LinearPlan {
  Plan g;            // token tile, issuers, rings (n_tiles1 / kst1 / S1 describe the one GEMM)
  int64_t M = 0;
  size_t off_status = 0, off_sorted = 0, off_expert = 0, off_scalars = 0, off_chunks = 0, off_xg = 0,
         off_xscale = 0, off_h = 0, total = 0;
};

qmoe_status validate_linear(const qmoe_linear* L) {
  if (L == nullptr) return QMOE_ERR_INVALID_ARG;
  if (L->N <= 0 || L->K <= 0) return QMOE_ERR_INVALID_ARG;
  if (L->N % 128 != 0 || L->K % 128 != 0) return QMOE_ERR_UNSUPPORTED;
  if (L->perm != nullptr && L->K > kMaxActOrderK) return QMOE_ERR_UNSUPPORTED;
  return validate_format(L->qt, L->group_size, L->act_dtype, L->scale_dtype, L->perm != nullptr);
}

qmoe_status make_linear_plan(const qmoe_linear* L, int64_t M, const qmoe_options* o, int sms, LinearPlan* lp) {
  qmoe_status st = validate_linear(L);
  if (st != QMOE_OK) return st;
  if (M < 0) return QMOE_ERR_INVALID_ARG;
  if (M >= (int64_t(1) << 31) - kAlignBlock) return QMOE_ERR_UNSUPPORTED;
  LinearPlan q;
  Plan& p = q.g;
  q.M = M;
  p.M = M;
  p.k = 1;
  p.P = M;
  // token tile: the power of two from 16 to 128 that holds all M rows, else 128
  int T = 16;
  while (T < 128 && T < M) T *= 2;
  if (o != nullptr && o->token_tile != 0) {
    if (o->token_tile < 16 || o->token_tile > kMaxTokenTile || o->token_tile % 16 != 0) return QMOE_ERR_INVALID_ARG;
    T = o->token_tile;
  }
  p.T = T;
  // (the dense linear layer runs on single CTAs)
  if (o != nullptr && (o->cta_pair < 0 || o->cta_pair > 2 || o->cta_pair == 1)) return QMOE_ERR_INVALID_ARG;
  p.stage_bytes = stage_bytes_of(L->qt, L->group_size);
  p.n_tiles1 = L->N / kTileRows;
  p.kst1 = L->K / kStageK;
  if ((st = size_gemm_rings(o, &p)) != QMOE_OK) return st;
  p.cap = (M + kAlignBlock - 1 + 15) / 16 * 16;
  p.nblocks = (p.cap + kAlignBlock - 1) / kAlignBlock;
  p.max_chunks = (p.cap + T - 1) / T + 1;
  const int64_t chunks = std::max<int64_t>(1, (M + T - 1) / T);
  const double epi = 4.0 + T / 8.0;
  p.S1 = choose_split(chunks * p.n_tiles1, p.kst1, sms, epi, 2.0 + 8.0 * M * L->N / 1.3e6, 0.9);
  if (o != nullptr && o->split1 != 0) {
    if (o->split1 < 1 || o->split1 > 64 || o->split1 > p.kst1) return QMOE_ERR_INVALID_ARG;
    p.S1 = o->split1;
  }
  size_t off = 0;
  q.off_status = off;   off += 256;
  q.off_sorted = off;   off += al256(p.cap * 4);
  q.off_expert = off;   off += al256(p.nblocks * 4);
  q.off_scalars = off;  off += 256;
  q.off_chunks = off;   off += al256(p.max_chunks * sizeof(Chunk));
  q.off_xg = off;       off += al256(static_cast<size_t>(p.cap) * L->K * 2);
  q.off_xscale = off;   off += al256(static_cast<size_t>(p.cap) * 4);
  q.off_h = off;        off += (p.S1 > 1) ? al256(static_cast<size_t>(p.S1) * p.cap * L->N * 4) : 0;
  q.total = off;
  *lp = q;
  return QMOE_OK;
}

qmoe_status linear_forward_impl(const qmoe_linear* L, const void* x, int64_t M, void* out, void* ws, size_t ws_bytes,
                                cudaStream_t stream, const qmoe_options* opts) {
  const int sms = current_sm_count();
  LinearPlan lp;
  qmoe_status st = make_linear_plan(L, M, opts, sms, &lp);
  if (st != QMOE_OK) return st;
  if (M == 0) return QMOE_OK;
  if (ws == nullptr || ws_bytes < lp.total) return QMOE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  const void* ptrs[] = {x, out, ws, L->w};
  for (const void* p : ptrs)
    if ((st = check_dev_ptr(p, dev)) != QMOE_OK) return st;
  const bool row_scales = has_row_scales(L->qt, L->group_size);
  if (row_scales && (st = check_dev_ptr(L->s, dev)) != QMOE_OK) return st;
  if (L->perm != nullptr && (st = check_dev_ptr(L->perm, dev)) != QMOE_OK) return st;
  if (!aligned(x, 256) || !aligned(out, 256) || !aligned(ws, 256) || !aligned(L->w, 256) ||
      (L->perm != nullptr && !aligned(L->perm, 16)) || (row_scales && !aligned(L->s, 16)))
    return QMOE_ERR_INVALID_ARG;
  const Plan& pl = lp.g;
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(base + lp.off_status);
  int32_t* sorted = reinterpret_cast<int32_t*>(base + lp.off_sorted);
  int32_t* expert = reinterpret_cast<int32_t*>(base + lp.off_expert);
  int32_t* npp = reinterpret_cast<int32_t*>(base + lp.off_scalars);
  int32_t* nch = npp + 1;
  Chunk* chunks = reinterpret_cast<Chunk*>(base + lp.off_chunks);
  void* xg = base + lp.off_xg;
  float* xscale = reinterpret_cast<float*>(base + lp.off_xscale);
  float* h = reinterpret_cast<float*>(base + lp.off_h);
  const bool bf16 = L->act_dtype == QMOE_BF16;
  const int P = static_cast<int>(M);
  // every row is "expert 0": the align kernel lays out rows 0..M-1 and the chunk table
  cudaError_t err;
  if (align_gather_small_fits(P, 1, kAlignBlock, L->K, L->perm != nullptr)) {
    err = launch_align_gather_small(nullptr, P, 1, kAlignBlock, pl.cap, sorted, expert, npp, pl.T, chunks, nch, status,
                                    x, bf16, L->perm, 1, L->K, pl.cap, xg, xscale, nullptr, sms, stream);
  } else {
    err = launch_align(nullptr, P, 1, kAlignBlock, pl.cap, sorted, expert, npp, pl.T, chunks, nch, status, stream);
    if (err == cudaSuccess)
      err = launch_gather(x, bf16, sorted, expert, npp, L->perm, P, 1, L->K, kAlignBlock, pl.cap, xg, xscale, nullptr,
                          sms, stream);
  }
  GemmParams g{};
  g.w = static_cast<const uint8_t*>(L->w);
  g.b = static_cast<const uint8_t*>(xg);
  g.b_unit_stride = pl.cap * 256;
  g.row_scale = row_scales ? L->s : nullptr;
  g.col_scale = xscale;
  g.chunks = chunks;
  g.n_chunks = nch;
  g.sorted_ids = sorted;
  g.topk_w = nullptr;
  g.status = status;
  g.n_tiles = pl.n_tiles1;
  g.k_groups = pl.kst1;
  g.split = pl.S1;
  g.token_tile = pl.T;
  g.acc_bufs = pl.acc_bufs;
  g.a_col0 = pl.a_col0;
  g.issuers = pl.issuers;
  g.w_stages = pl.w_stages;
  g.ab_stages = pl.ab_stages;
  g.b_stages = pl.b_stages;
  g.dq_sets = pl.dq_sets;
  g.fault_injection = 0;
  g.stage_bytes = pl.stage_bytes;
  g.P = P;
  g.chunk_group = chunk_raster(P, 1, pl.T, L->K);
  g.inter_ld = 0;
  g.w_shared = (opts != nullptr && opts->weight_l2 != 0) ? (opts->weight_l2 == 1) : (M > pl.T);
  g.out_bf16 = bf16 ? 1 : 0;
  if (pl.S1 == 1) {
    g.epi_mode = kEpiLinearOut;
    g.out = out;
    g.out_ld = L->N;
    g.out_split_stride = 0;
  } else {
    g.epi_mode = kEpiPartialRows;
    g.out = h;
    g.out_ld = L->N;
    g.out_split_stride = pl.cap * static_cast<int64_t>(L->N);
  }
  const int64_t items = pl.max_chunks * pl.n_tiles1 * pl.S1;
  const int grid = static_cast<int>(std::min<int64_t>(sms, items));
  if (err == cudaSuccess) err = launch_gemm(kind_of(L->qt, L->group_size), bf16, g, grid, stream);
  if (err == cudaSuccess && pl.S1 > 1) err = launch_linear_reduce(h, pl.S1, pl.cap, M, L->N, bf16, out, sms, stream);
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

size_t host_staging_bytes(const qmoe_layer* L, int64_t M, int32_t k) {
  return 2 * al256(static_cast<size_t>(M) * L->H * 2) + 2 * al256(static_cast<size_t>(M) * k * 4);
}

// ---------------------------------------------------------------------------
// packing
// ---------------------------------------------------------------------------
// Stable order of the K positions by group; checks that each group has exactly 128 members.
bool sorted_by_group(const int32_t* g, int K, std::vector<int32_t>& perm) {
  const int ng = K / 128;
  std::vector<int> count(ng, 0);
  for (int kk = 0; kk < K; ++kk) {
    if (g[kk] < 0 || g[kk] >= ng) return false;
    ++count[g[kk]];
  }
  for (int c : count)
    if (c != 128) return false;
  perm.resize(K);
  std::vector<int> cur(ng);
  for (int i = 0; i < ng; ++i) cur[i] = i * 128;
  for (int kk = 0; kk < K; ++kk) perm[cur[g[kk]]++] = kk;
  return true;
}

// Packed row r of W13 tile t -> canonical row: rows 2j / 2j+1 of the tile are
// gate / up of intermediate channel 64t + j in the new (act-order sorted) order.
inline int w13_canon_row(int t, int r, int I, const int32_t* perm2) {
  const int jn = 64 * t + (r >> 1);
  const int j = perm2 ? perm2[jn] : jn;
  return (r & 1) ? I + j : j;
}

// int4 tile stage: 4 chunks x 128 rows x 16 B, then 128 x 2 B scales (and, with
// zero points, 128 x 1 B zero points).
// Chunk c of a row holds sorted K = 32c..32c+31; word j of it holds
// K = 32c+8j .. +7 with nibble i <- K 32c+8j+2i and nibble i+4 <- K 32c+8j+2i+1.
// s (and z) are [groups][rows]; with one group over all of K (channel-wise) the
// row's one scale is repeated in every stage block.
void pack_int4_matrix(const uint8_t* q, const uint16_t* s, const uint8_t* z, bool channel_wise, int rows, int K,
                      int I_for_w13, const int32_t* perm2_rows, const int32_t* kperm, uint8_t* out,
                      std::atomic<bool>& bad) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = z ? kInt4ZpStageBytes : kInt4StageBytes;
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      uint8_t* blk = out + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      const int grp = channel_wise ? 0 : ks;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, perm2_rows) : t * 128 + r;
        const uint8_t* qrow = q + static_cast<size_t>(cr) * K;
        for (int c = 0; c < 4; ++c)
          for (int j = 0; j < 4; ++j) {
            uint32_t word = 0;
            for (int i = 0; i < 4; ++i) {
              const int k0 = ks * 128 + 32 * c + 8 * j + 2 * i;
              const int c0 = kperm ? kperm[k0] : k0;
              const int c1 = kperm ? kperm[k0 + 1] : k0 + 1;
              const uint8_t a = qrow[c0], b = qrow[c1];
              if (a > 15 || b > 15) bad = true;
              word |= static_cast<uint32_t>(a & 15) << (4 * i);
              word |= static_cast<uint32_t>(b & 15) << (4 * (i + 4));
            }
            uint8_t* dst = blk + (c * 128 + r) * 16 + j * 4;
            dst[0] = word & 0xFF;
            dst[1] = (word >> 8) & 0xFF;
            dst[2] = (word >> 16) & 0xFF;
            dst[3] = (word >> 24) & 0xFF;
          }
        const uint16_t sb = s[static_cast<size_t>(grp) * rows + cr];
        blk[8192 + r * 2] = sb & 0xFF;
        blk[8192 + r * 2 + 1] = sb >> 8;
        if (z) {
          const uint8_t zv = z[static_cast<size_t>(grp) * rows + cr];
          if (zv > 15) bad = true;
          blk[8448 + r] = zv;
        }
      }
    }
}

void unpack_int4_matrix(const uint8_t* in, bool zp, bool channel_wise, int rows, int K, int I_for_w13,
                        const int32_t* perm2_rows, const int32_t* kperm, uint8_t* q, uint16_t* s, uint8_t* z) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = zp ? kInt4ZpStageBytes : kInt4StageBytes;
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      const uint8_t* blk = in + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      const int grp = channel_wise ? 0 : ks;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, perm2_rows) : t * 128 + r;
        uint8_t* qrow = q + static_cast<size_t>(cr) * K;
        for (int c = 0; c < 4; ++c)
          for (int j = 0; j < 4; ++j) {
            const uint8_t* src = blk + (c * 128 + r) * 16 + j * 4;
            const uint32_t word = src[0] | (src[1] << 8) | (src[2] << 16) | (static_cast<uint32_t>(src[3]) << 24);
            for (int i = 0; i < 4; ++i) {
              const int k0 = ks * 128 + 32 * c + 8 * j + 2 * i;
              qrow[kperm ? kperm[k0] : k0] = (word >> (4 * i)) & 15;
              qrow[kperm ? kperm[k0 + 1] : k0 + 1] = (word >> (4 * (i + 4))) & 15;
            }
          }
        s[static_cast<size_t>(grp) * rows + cr] = static_cast<uint16_t>(blk[8192 + r * 2] | (blk[8192 + r * 2 + 1] << 8));
        if (zp && z) z[static_cast<size_t>(grp) * rows + cr] = blk[8448 + r];
      }
    }
}

// 2:4 position words in the order the tensor core's structured-sparse MMA reads
// them from tensor memory.  nib[r * 32 + g] = i0 | i1 << 2: the kept channels of
// group g (4 input channels) of row r of a 128-row tile, one 128-K stage.  Sparse
// MMA k (0..3) covers groups 8k .. 8k+7 as two sub-blocks of 4 groups; the TMEM
// lane L = 16b + 8s + i holds, for MMA k, sub-block s of row 16b + i in bits 0-15
// and sub-block s of row 16b + 8 + i in bits 16-31, 4 bits per group in ascending
// order (measured on GB300 by a self-checking probe with one-hot B operands).  The
// word of lane L for MMA k sits at byte (k / 2) * 1024 + L * 8 + (k % 2) * 4 of the
// 2048-byte position area, so the thread of lane L loads 8 bytes per K half.
void store_sparse_positions(const uint8_t* nib, uint8_t* posarea) {
  for (int L = 0; L < 128; ++L) {
    const int b = L / 16, sb = (L / 8) % 2, i = L % 8;
    const int r0 = 16 * b + i, r1 = 16 * b + 8 + i;
    for (int k = 0; k < 4; ++k) {
      uint32_t w = 0;
      for (int t = 0; t < 4; ++t) {
        const int g = 8 * k + 4 * sb + t;
        w |= static_cast<uint32_t>(nib[r0 * 32 + g]) << (4 * t);
        w |= static_cast<uint32_t>(nib[r1 * 32 + g]) << (16 + 4 * t);
      }
      uint8_t* dst = posarea + (k / 2) * 1024 + L * 8 + (k % 2) * 4;
      for (int x = 0; x < 4; ++x) dst[x] = static_cast<uint8_t>(w >> (8 * x));
    }
  }
}

void load_sparse_positions(const uint8_t* posarea, uint8_t* nib) {
  for (int L = 0; L < 128; ++L) {
    const int b = L / 16, sb = (L / 8) % 2, i = L % 8;
    const int r0 = 16 * b + i, r1 = 16 * b + 8 + i;
    for (int k = 0; k < 4; ++k) {
      const uint8_t* src = posarea + (k / 2) * 1024 + L * 8 + (k % 2) * 4;
      const uint32_t w = src[0] | (src[1] << 8) | (src[2] << 16) | (static_cast<uint32_t>(src[3]) << 24);
      for (int t = 0; t < 4; ++t) {
        const int g = 8 * k + 4 * sb + t;
        nib[r0 * 32 + g] = static_cast<uint8_t>((w >> (4 * t)) & 15);
        nib[r1 * 32 + g] = static_cast<uint8_t>((w >> (16 + 4 * t)) & 15);
      }
    }
  }
}

// 2:4-sparse int4 tile stage (6400 B): kept codes [half][row][16 B], the 2048-byte
// position area (store_sparse_positions), then 128 x 2 B scales.  Half h covers
// K = 64h .. 64h+63, 16 groups of 4 channels.  Word j of a row's 16 code bytes
// holds groups 4j..4j+3 of the half: nibble i <- the first kept code of group
// 4j+i, nibble i+4 <- the second.  Per group the kept channels are those with a
// code other than 8, padded with the lowest remaining channels (positions
// i0 < i1); more than 2 sets `bad`.
void pack_int4_24_matrix(const uint8_t* q, const uint16_t* s, bool channel_wise, int rows, int K, int I_for_w13,
                         uint8_t* out, std::atomic<bool>& bad) {
  const int n_tiles = rows / 128, kst = K / 128;
  std::vector<uint8_t> nib(128 * 32);
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      uint8_t* blk = out + (static_cast<size_t>(t) * kst + ks) * kInt4SparseStageBytes;
      const int grp = channel_wise ? 0 : ks;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        const uint8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int h = 0; h < 2; ++h) {
          uint8_t v0[16], v1[16];
          for (int g = 0; g < 16; ++g) {
            const uint8_t* c4 = qrow + 64 * h + 4 * g;
            int keep[4], n = 0;
            for (int i = 0; i < 4; ++i) {
              if (c4[i] > 15) bad = true;
              if (c4[i] != 8) {
                if (n == 2) bad = true;
                else keep[n++] = i;
              }
            }
            for (int i = 0; i < 4 && n < 2; ++i)
              if (c4[i] == 8 && (n == 0 || keep[0] != i)) keep[n++] = i;
            if (keep[0] > keep[1]) std::swap(keep[0], keep[1]);
            v0[g] = c4[keep[0]] & 15;
            v1[g] = c4[keep[1]] & 15;
            nib[r * 32 + 16 * h + g] = static_cast<uint8_t>(keep[0] | (keep[1] << 2));
          }
          uint8_t* vdst = blk + (h * 128 + r) * 16;
          for (int j = 0; j < 4; ++j) {
            uint32_t word = 0;
            for (int i = 0; i < 4; ++i) {
              word |= static_cast<uint32_t>(v0[4 * j + i]) << (4 * i);
              word |= static_cast<uint32_t>(v1[4 * j + i]) << (4 * (i + 4));
            }
            for (int b = 0; b < 4; ++b) vdst[4 * j + b] = static_cast<uint8_t>(word >> (8 * b));
          }
        }
        const uint16_t sb = s[static_cast<size_t>(grp) * rows + cr];
        blk[6144 + r * 2] = sb & 0xFF;
        blk[6144 + r * 2 + 1] = sb >> 8;
      }
      store_sparse_positions(nib.data(), blk + 4096);
    }
}

void unpack_int4_24_matrix(const uint8_t* in, bool channel_wise, int rows, int K, int I_for_w13, uint8_t* q,
                           uint16_t* s) {
  const int n_tiles = rows / 128, kst = K / 128;
  std::vector<uint8_t> nib(128 * 32);
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      const uint8_t* blk = in + (static_cast<size_t>(t) * kst + ks) * kInt4SparseStageBytes;
      const int grp = channel_wise ? 0 : ks;
      load_sparse_positions(blk + 4096, nib.data());
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        uint8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int h = 0; h < 2; ++h) {
          const uint8_t* vsrc = blk + (h * 128 + r) * 16;
          for (int g = 0; g < 16; ++g) {
            const int j = g / 4, i = g % 4;
            const uint32_t word = vsrc[4 * j] | (vsrc[4 * j + 1] << 8) | (vsrc[4 * j + 2] << 16) |
                                  (static_cast<uint32_t>(vsrc[4 * j + 3]) << 24);
            const int p = nib[r * 32 + 16 * h + g];
            uint8_t* c4 = qrow + 64 * h + 4 * g;
            for (int x = 0; x < 4; ++x) c4[x] = 8;
            c4[p & 3] = (word >> (4 * i)) & 15;
            c4[p >> 2] = (word >> (4 * (i + 4))) & 15;
          }
        }
        s[static_cast<size_t>(grp) * rows + cr] = static_cast<uint16_t>(blk[6144 + r * 2] | (blk[6144 + r * 2 + 1] << 8));
      }
    }
}

// int8 tile stage: 8 chunks x 128 rows x 16 B; chunk c holds K = 16c..16c+15 in
// byte order.  With group scales (s [groups][rows], 16-bit) 128 x 2 B scales follow.
void pack_int8_matrix(const int8_t* q, const uint16_t* s, int rows, int K, int I_for_w13, uint8_t* out,
                      std::atomic<bool>& bad) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = s ? kInt8GroupStageBytes : kInt8StageBytes;
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      uint8_t* blk = out + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        const int8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int c = 0; c < 8; ++c)
          for (int b = 0; b < 16; ++b) {
            const int8_t v = qrow[16 * c + b];
            if (v == -128) bad = true;
            blk[(c * 128 + r) * 16 + b] = static_cast<uint8_t>(v);
          }
        if (s) {
          const uint16_t sb = s[static_cast<size_t>(ks) * rows + cr];
          blk[16384 + r * 2] = sb & 0xFF;
          blk[16384 + r * 2 + 1] = sb >> 8;
        }
      }
    }
}

void unpack_int8_matrix(const uint8_t* in, bool grouped, int rows, int K, int I_for_w13, int8_t* q, uint16_t* s) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = grouped ? kInt8GroupStageBytes : kInt8StageBytes;
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      const uint8_t* blk = in + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        int8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int c = 0; c < 8; ++c)
          for (int b = 0; b < 16; ++b) qrow[16 * c + b] = static_cast<int8_t>(blk[(c * 128 + r) * 16 + b]);
        if (grouped && s)
          s[static_cast<size_t>(ks) * rows + cr] = static_cast<uint16_t>(blk[16384 + r * 2] | (blk[16384 + r * 2 + 1] << 8));
      }
    }
}

// 2:4-sparse int8 tile stage: kept codes [half][row][32 B], the 2048-byte
// position area at 8192 (store_sparse_positions), then (with group scales) 128 x
// 2 B scales at 10240.  Half h covers K = 64h .. 64h+63, 16 groups of 4 channels;
// byte 2g + v of a row's 32 code bytes is kept code v of group g.  The kept
// channels are those with a non-zero code, padded with the lowest remaining
// channels; more than 2 non-zero codes, or a code of -128, sets `bad`.
void pack_int8_24_matrix(const int8_t* q, const uint16_t* s, int rows, int K, int I_for_w13, uint8_t* out,
                         std::atomic<bool>& bad) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = s ? kInt8SparseGroupStageBytes : kInt8SparseStageBytes;
  std::vector<uint8_t> nib(128 * 32);
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      uint8_t* blk = out + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        const int8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int h = 0; h < 2; ++h) {
          uint8_t* vdst = blk + (h * 128 + r) * 32;
          for (int g = 0; g < 16; ++g) {
            const int8_t* c4 = qrow + 64 * h + 4 * g;
            int keep[4], n = 0;
            for (int i = 0; i < 4; ++i) {
              if (c4[i] == -128) bad = true;
              if (c4[i] != 0) {
                if (n == 2) bad = true;
                else keep[n++] = i;
              }
            }
            for (int i = 0; i < 4 && n < 2; ++i)
              if (c4[i] == 0 && (n == 0 || keep[0] != i)) keep[n++] = i;
            if (keep[0] > keep[1]) std::swap(keep[0], keep[1]);
            vdst[2 * g] = static_cast<uint8_t>(c4[keep[0]]);
            vdst[2 * g + 1] = static_cast<uint8_t>(c4[keep[1]]);
            nib[r * 32 + 16 * h + g] = static_cast<uint8_t>(keep[0] | (keep[1] << 2));
          }
        }
        if (s) {
          const uint16_t sb = s[static_cast<size_t>(ks) * rows + cr];
          blk[10240 + r * 2] = sb & 0xFF;
          blk[10240 + r * 2 + 1] = sb >> 8;
        }
      }
      store_sparse_positions(nib.data(), blk + 8192);
    }
}

void unpack_int8_24_matrix(const uint8_t* in, bool grouped, int rows, int K, int I_for_w13, int8_t* q, uint16_t* s) {
  const int n_tiles = rows / 128, kst = K / 128;
  const size_t blk_bytes = grouped ? kInt8SparseGroupStageBytes : kInt8SparseStageBytes;
  std::vector<uint8_t> nib(128 * 32);
  for (int t = 0; t < n_tiles; ++t)
    for (int ks = 0; ks < kst; ++ks) {
      const uint8_t* blk = in + (static_cast<size_t>(t) * kst + ks) * blk_bytes;
      load_sparse_positions(blk + 8192, nib.data());
      for (int r = 0; r < 128; ++r) {
        const int cr = I_for_w13 > 0 ? w13_canon_row(t, r, I_for_w13, nullptr) : t * 128 + r;
        int8_t* qrow = q + static_cast<size_t>(cr) * K + ks * 128;
        for (int h = 0; h < 2; ++h) {
          const uint8_t* vsrc = blk + (h * 128 + r) * 32;
          for (int g = 0; g < 16; ++g) {
            const int p = nib[r * 32 + 16 * h + g];
            int8_t* c4 = qrow + 64 * h + 4 * g;
            for (int x = 0; x < 4; ++x) c4[x] = 0;
            c4[p & 3] = static_cast<int8_t>(vsrc[2 * g]);
            c4[p >> 2] = static_cast<int8_t>(vsrc[2 * g + 1]);
          }
        }
        if (grouped && s)
          s[static_cast<size_t>(ks) * rows + cr] = static_cast<uint16_t>(blk[10240 + r * 2] | (blk[10240 + r * 2 + 1] << 8));
      }
    }
}

bool pack_dims_ok(int32_t E, int32_t H, int32_t I) {
  return E >= 1 && E <= 1024 && H > 0 && I > 0 && H % 128 == 0 && I % 128 == 0;
}

}  // namespace

qmoe_status forward_into_workspace(const qmoe_layer* layer, const void* x, int64_t M, const int32_t* topk_ids,
                                   const float* topk_weights, int32_t top_k, void* out, void* ws, size_t ws_bytes,
                                   cudaStream_t stream) {
  return forward_impl(layer, x, M, topk_ids, topk_weights, top_k, out, ws, ws_bytes, stream, nullptr);
}

}  // namespace qmoe

using namespace qmoe;

extern "C" {

int32_t qmoe_abi_version(void) { return QMOE_ABI_VERSION; }

const char* qmoe_status_string(qmoe_status s) {
  switch (s) {
    case QMOE_OK: return "ok";
    case QMOE_ERR_INVALID_ARG: return "invalid argument";
    case QMOE_ERR_UNSUPPORTED: return "unsupported shape, group size or type combination";
    case QMOE_ERR_DEVICE_MISMATCH: return "pointer is not device memory of the current device";
    case QMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case QMOE_ERR_CUDA: return "CUDA runtime or launch error";
    case QMOE_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    case QMOE_ERR_BAD_EXPERT_ID: return "a top-k expert id is outside [0, E)";
  }
  return "unknown status";
}

size_t qmoe_packed_bytes(qmoe_quant_type qt, int32_t E, int32_t rows, int32_t K, int32_t group_size) {
  if (E < 1 || rows <= 0 || K <= 0 || rows % 128 != 0 || K % 128 != 0) return 0;
  const size_t tiles = static_cast<size_t>(E) * (rows / 128) * (K / 128);
  const bool g128_or_cw = group_size == 128 || group_size == -1;
  if (qt == QMOE_INT4_GROUP && g128_or_cw) return tiles * kInt4StageBytes;
  if (qt == QMOE_INT4_GROUP_ZP && g128_or_cw) return tiles * kInt4ZpStageBytes;
  if (qt == QMOE_INT8_PER_COL && group_size == -1) return tiles * kInt8StageBytes;
  if (qt == QMOE_INT8_GROUP && group_size == 128) return tiles * kInt8GroupStageBytes;
  if (qt == QMOE_INT4_GROUP_24 && g128_or_cw) return tiles * kInt4SparseStageBytes;
  if (qt == QMOE_INT8_24 && group_size == -1) return tiles * kInt8SparseStageBytes;
  if (qt == QMOE_INT8_24 && group_size == 128) return tiles * kInt8SparseGroupStageBytes;
  return 0;
}

}  // extern "C"

namespace {

qmoe_status pack_int4_any(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                          const uint8_t* q13, const uint16_t* s13, const uint8_t* z13, const int32_t* g13,
                          const uint8_t* q2, const uint16_t* s2, const uint8_t* z2, const int32_t* g2,
                          void* w13_packed, void* w2_packed, int32_t* perm13_out) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  if (group_size == -1 && (g13 || g2)) return QMOE_ERR_UNSUPPORTED;
  if (scale_dtype != QMOE_F16 && scale_dtype != QMOE_BF16) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed || (g13 && !perm13_out)) return QMOE_ERR_INVALID_ARG;
  const bool zp = z13 != nullptr;
  if (zp != (z2 != nullptr)) return QMOE_ERR_INVALID_ARG;
  const bool cw = group_size == -1;
  const qmoe_quant_type qt = zp ? QMOE_INT4_GROUP_ZP : QMOE_INT4_GROUP;
  std::atomic<bool> bad{false}, badg{false};
  const size_t b13 = qmoe_packed_bytes(qt, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(qt, 1, H, I, group_size);
  const size_t ng13 = cw ? 1 : H / 128, ng2 = cw ? 1 : I / 128;
  parallel_for(E, [&](int64_t e) {
    std::vector<int32_t> p13, p2;
    if (g13 && !sorted_by_group(g13 + e * H, H, p13)) { badg = true; return; }
    if (g2 && !sorted_by_group(g2 + e * I, I, p2)) { badg = true; return; }
    if (g13) std::memcpy(perm13_out + e * H, p13.data(), sizeof(int32_t) * H);
    pack_int4_matrix(q13 + static_cast<size_t>(e) * 2 * I * H, s13 + e * ng13 * 2 * I,
                     zp ? z13 + e * ng13 * 2 * I : nullptr, cw, 2 * I, H, I, g2 ? p2.data() : nullptr,
                     g13 ? p13.data() : nullptr, static_cast<uint8_t*>(w13_packed) + e * b13, bad);
    pack_int4_matrix(q2 + static_cast<size_t>(e) * H * I, s2 + e * ng2 * H, zp ? z2 + e * ng2 * H : nullptr, cw, H,
                     I, 0, nullptr, g2 ? p2.data() : nullptr, static_cast<uint8_t*>(w2_packed) + e * b2, bad);
  });
  if (badg) return QMOE_ERR_UNSUPPORTED;
  if (bad) return QMOE_ERR_INVALID_ARG;
  return QMOE_OK;
}

qmoe_status unpack_int4_any(int32_t E, int32_t H, int32_t I, int32_t group_size, bool zp, const void* w13_packed,
                            const void* w2_packed, const int32_t* g13, const int32_t* g2, uint8_t* q13,
                            uint16_t* s13, uint8_t* z13, uint8_t* q2, uint16_t* s2, uint8_t* z2) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  if (group_size == -1 && (g13 || g2)) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed || (zp && (!z13 || !z2))) return QMOE_ERR_INVALID_ARG;
  const bool cw = group_size == -1;
  const qmoe_quant_type qt = zp ? QMOE_INT4_GROUP_ZP : QMOE_INT4_GROUP;
  std::atomic<bool> badg{false};
  const size_t b13 = qmoe_packed_bytes(qt, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(qt, 1, H, I, group_size);
  const size_t ng13 = cw ? 1 : H / 128, ng2 = cw ? 1 : I / 128;
  parallel_for(E, [&](int64_t e) {
    std::vector<int32_t> p13, p2;
    if (g13 && !sorted_by_group(g13 + e * H, H, p13)) { badg = true; return; }
    if (g2 && !sorted_by_group(g2 + e * I, I, p2)) { badg = true; return; }
    unpack_int4_matrix(static_cast<const uint8_t*>(w13_packed) + e * b13, zp, cw, 2 * I, H, I,
                       g2 ? p2.data() : nullptr, g13 ? p13.data() : nullptr, q13 + static_cast<size_t>(e) * 2 * I * H,
                       s13 + e * ng13 * 2 * I, zp ? z13 + e * ng13 * 2 * I : nullptr);
    unpack_int4_matrix(static_cast<const uint8_t*>(w2_packed) + e * b2, zp, cw, H, I, 0, nullptr,
                       g2 ? p2.data() : nullptr, q2 + static_cast<size_t>(e) * H * I, s2 + e * ng2 * H,
                       zp ? z2 + e * ng2 * H : nullptr);
  });
  return badg ? QMOE_ERR_UNSUPPORTED : QMOE_OK;
}

}  // namespace

extern "C" {

qmoe_status qmoe_pack_int4(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                           const uint8_t* q13, const uint16_t* s13, const int32_t* g13, const uint8_t* q2,
                           const uint16_t* s2, const int32_t* g2, void* w13_packed, void* w2_packed,
                           int32_t* perm13_out) {
  return pack_int4_any(E, H, I, group_size, scale_dtype, q13, s13, nullptr, g13, q2, s2, nullptr, g2, w13_packed,
                       w2_packed, perm13_out);
}

qmoe_status qmoe_unpack_int4(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                             const void* w2_packed, const int32_t* g13, const int32_t* g2, uint8_t* q13,
                             uint16_t* s13, uint8_t* q2, uint16_t* s2) {
  return unpack_int4_any(E, H, I, group_size, false, w13_packed, w2_packed, g13, g2, q13, s13, nullptr, q2, s2,
                         nullptr);
}

qmoe_status qmoe_pack_int4_zp(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const uint8_t* q13, const uint16_t* s13, const uint8_t* z13, const int32_t* g13,
                              const uint8_t* q2, const uint16_t* s2, const uint8_t* z2, const int32_t* g2,
                              void* w13_packed, void* w2_packed, int32_t* perm13_out) {
  if (!z13 || !z2) return QMOE_ERR_INVALID_ARG;
  return pack_int4_any(E, H, I, group_size, scale_dtype, q13, s13, z13, g13, q2, s2, z2, g2, w13_packed, w2_packed,
                       perm13_out);
}

qmoe_status qmoe_unpack_int4_zp(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                                const void* w2_packed, const int32_t* g13, const int32_t* g2, uint8_t* q13,
                                uint16_t* s13, uint8_t* z13, uint8_t* q2, uint16_t* s2, uint8_t* z2) {
  return unpack_int4_any(E, H, I, group_size, true, w13_packed, w2_packed, g13, g2, q13, s13, z13, q2, s2, z2);
}

qmoe_status qmoe_pack_int8(int32_t E, int32_t H, int32_t I, const int8_t* q13, const float* s13, const int8_t* q2,
                           const float* s2, void* w13_packed, float* s13_packed, void* w2_packed, float* s2_packed) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !s13_packed || !w2_packed || !s2_packed)
    return QMOE_ERR_INVALID_ARG;
  std::atomic<bool> bad{false};
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_PER_COL, 1, 2 * I, H, -1);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_PER_COL, 1, H, I, -1);
  parallel_for(E, [&](int64_t e) {
    pack_int8_matrix(q13 + static_cast<size_t>(e) * 2 * I * H, nullptr, 2 * I, H, I,
                     static_cast<uint8_t*>(w13_packed) + e * b13, bad);
    pack_int8_matrix(q2 + static_cast<size_t>(e) * H * I, nullptr, H, I, 0,
                     static_cast<uint8_t*>(w2_packed) + e * b2, bad);
    for (int t = 0; t < 2 * I / 128; ++t)
      for (int r = 0; r < 128; ++r)
        s13_packed[static_cast<size_t>(e) * 2 * I + t * 128 + r] = s13[static_cast<size_t>(e) * 2 * I + w13_canon_row(t, r, I, nullptr)];
    std::memcpy(s2_packed + static_cast<size_t>(e) * H, s2 + static_cast<size_t>(e) * H, sizeof(float) * H);
  });
  return bad ? QMOE_ERR_INVALID_ARG : QMOE_OK;
}

qmoe_status qmoe_unpack_int8(int32_t E, int32_t H, int32_t I, const void* w13_packed, const float* s13_packed,
                             const void* w2_packed, const float* s2_packed, int8_t* q13, float* s13, int8_t* q2,
                             float* s2) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !s13_packed || !w2_packed || !s2_packed)
    return QMOE_ERR_INVALID_ARG;
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_PER_COL, 1, 2 * I, H, -1);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_PER_COL, 1, H, I, -1);
  parallel_for(E, [&](int64_t e) {
    unpack_int8_matrix(static_cast<const uint8_t*>(w13_packed) + e * b13, false, 2 * I, H, I,
                       q13 + static_cast<size_t>(e) * 2 * I * H, nullptr);
    unpack_int8_matrix(static_cast<const uint8_t*>(w2_packed) + e * b2, false, H, I, 0,
                       q2 + static_cast<size_t>(e) * H * I, nullptr);
    for (int t = 0; t < 2 * I / 128; ++t)
      for (int r = 0; r < 128; ++r)
        s13[static_cast<size_t>(e) * 2 * I + w13_canon_row(t, r, I, nullptr)] = s13_packed[static_cast<size_t>(e) * 2 * I + t * 128 + r];
    std::memcpy(s2 + static_cast<size_t>(e) * H, s2_packed + static_cast<size_t>(e) * H, sizeof(float) * H);
  });
  return QMOE_OK;
}

qmoe_status qmoe_pack_int8_group(int32_t E, int32_t H, int32_t I, qmoe_dtype scale_dtype, const int8_t* q13,
                                 const uint16_t* s13, const int8_t* q2, const uint16_t* s2, void* w13_packed,
                                 void* w2_packed) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (scale_dtype != QMOE_F16 && scale_dtype != QMOE_BF16) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed) return QMOE_ERR_INVALID_ARG;
  std::atomic<bool> bad{false};
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_GROUP, 1, 2 * I, H, 128);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_GROUP, 1, H, I, 128);
  parallel_for(E, [&](int64_t e) {
    pack_int8_matrix(q13 + static_cast<size_t>(e) * 2 * I * H, s13 + static_cast<size_t>(e) * (H / 128) * 2 * I,
                     2 * I, H, I, static_cast<uint8_t*>(w13_packed) + e * b13, bad);
    pack_int8_matrix(q2 + static_cast<size_t>(e) * H * I, s2 + static_cast<size_t>(e) * (I / 128) * H, H, I, 0,
                     static_cast<uint8_t*>(w2_packed) + e * b2, bad);
  });
  return bad ? QMOE_ERR_INVALID_ARG : QMOE_OK;
}

qmoe_status qmoe_unpack_int8_group(int32_t E, int32_t H, int32_t I, const void* w13_packed, const void* w2_packed,
                                   int8_t* q13, uint16_t* s13, int8_t* q2, uint16_t* s2) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed) return QMOE_ERR_INVALID_ARG;
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_GROUP, 1, 2 * I, H, 128);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_GROUP, 1, H, I, 128);
  parallel_for(E, [&](int64_t e) {
    unpack_int8_matrix(static_cast<const uint8_t*>(w13_packed) + e * b13, true, 2 * I, H, I,
                       q13 + static_cast<size_t>(e) * 2 * I * H, s13 + static_cast<size_t>(e) * (H / 128) * 2 * I);
    unpack_int8_matrix(static_cast<const uint8_t*>(w2_packed) + e * b2, true, H, I, 0,
                       q2 + static_cast<size_t>(e) * H * I, s2 + static_cast<size_t>(e) * (I / 128) * H);
  });
  return QMOE_OK;
}

qmoe_status qmoe_pack_int4_24(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const uint8_t* q13, const uint16_t* s13, const uint8_t* q2, const uint16_t* s2,
                              void* w13_packed, void* w2_packed) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  if (scale_dtype != QMOE_F16 && scale_dtype != QMOE_BF16) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed) return QMOE_ERR_INVALID_ARG;
  const bool cw = group_size == -1;
  const size_t b13 = qmoe_packed_bytes(QMOE_INT4_GROUP_24, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT4_GROUP_24, 1, H, I, group_size);
  const size_t ng13 = cw ? 1 : H / 128, ng2 = cw ? 1 : I / 128;
  std::atomic<bool> bad{false};
  parallel_for(E, [&](int64_t e) {
    pack_int4_24_matrix(q13 + static_cast<size_t>(e) * 2 * I * H, s13 + e * ng13 * 2 * I, cw, 2 * I, H, I,
                        static_cast<uint8_t*>(w13_packed) + e * b13, bad);
    pack_int4_24_matrix(q2 + static_cast<size_t>(e) * H * I, s2 + e * ng2 * H, cw, H, I, 0,
                        static_cast<uint8_t*>(w2_packed) + e * b2, bad);
  });
  return bad ? QMOE_ERR_INVALID_ARG : QMOE_OK;
}

qmoe_status qmoe_unpack_int4_24(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                                const void* w2_packed, uint8_t* q13, uint16_t* s13, uint8_t* q2, uint16_t* s2) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed) return QMOE_ERR_INVALID_ARG;
  const bool cw = group_size == -1;
  const size_t b13 = qmoe_packed_bytes(QMOE_INT4_GROUP_24, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT4_GROUP_24, 1, H, I, group_size);
  const size_t ng13 = cw ? 1 : H / 128, ng2 = cw ? 1 : I / 128;
  parallel_for(E, [&](int64_t e) {
    unpack_int4_24_matrix(static_cast<const uint8_t*>(w13_packed) + e * b13, cw, 2 * I, H, I,
                          q13 + static_cast<size_t>(e) * 2 * I * H, s13 + e * ng13 * 2 * I);
    unpack_int4_24_matrix(static_cast<const uint8_t*>(w2_packed) + e * b2, cw, H, I, 0,
                          q2 + static_cast<size_t>(e) * H * I, s2 + e * ng2 * H);
  });
  return QMOE_OK;
}

qmoe_status qmoe_moe_align(const int32_t* topk_ids, int64_t M, int32_t top_k, int32_t E, int32_t block,
                           int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded, int64_t capacity,
                           void* stream) {
  if (M < 0 || top_k < 1 || E < 1 || E > 1024 || block < 1 || block > 256) return QMOE_ERR_INVALID_ARG;
  const int64_t P = M * top_k;
  if (P >= (int64_t(1) << 31) - int64_t(E) * block) return QMOE_ERR_UNSUPPORTED;
  if (capacity < P + static_cast<int64_t>(E) * (block - 1)) return QMOE_ERR_INVALID_ARG;
  if (!sorted_ids || !expert_ids || !num_post_padded || (P > 0 && !topk_ids)) return QMOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  qmoe_status st;
  if (P > 0 && (st = check_dev_ptr(topk_ids, dev)) != QMOE_OK) return st;
  if ((st = check_dev_ptr(sorted_ids, dev)) != QMOE_OK) return st;
  if ((st = check_dev_ptr(expert_ids, dev)) != QMOE_OK) return st;
  if ((st = check_dev_ptr(num_post_padded, dev)) != QMOE_OK) return st;
  const cudaError_t err = launch_align(topk_ids, static_cast<int32_t>(P), E, block, capacity, sorted_ids, expert_ids,
                                       num_post_padded, 0, nullptr, nullptr, nullptr,
                                       static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

size_t qmoe_workspace_size_ex(const qmoe_layer* layer, int64_t M, int32_t top_k, const qmoe_options* opts) {
  Plan pl;
  if (make_plan(layer, M, top_k, opts, current_sm_count(), &pl) != QMOE_OK) return 0;
  return pl.total;
}

qmoe_status qmoe_describe_plan(const qmoe_layer* layer, int64_t M, int32_t top_k, const qmoe_options* opts,
                               int32_t num_sms, qmoe_plan_info* info) {
  if (info == nullptr || num_sms < 0) return QMOE_ERR_INVALID_ARG;
  Plan pl;
  const qmoe_status st = make_plan(layer, M, top_k, opts, num_sms > 0 ? num_sms : current_sm_count(), &pl);
  if (st != QMOE_OK) return st;
  *info = qmoe_plan_info{};
  info->token_tile = pl.T;
  info->issuers = pl.issuers;
  info->acc_bufs = pl.acc_bufs;
  info->split1 = pl.S1;
  info->split2 = pl.S2;
  info->w_stages = pl.w_stages;
  info->ab_stages = pl.ab_stages;
  info->b_stages = pl.b_stages;
  info->dq_sets = pl.dq_sets;
  info->cta_pair = pl.pair;
  info->cta_pair_down = pl.r2.pair;
  info->stage_bytes = pl.stage_bytes;
  info->workspace_bytes = static_cast<int64_t>(pl.total);
  return QMOE_OK;
}

size_t qmoe_workspace_size(const qmoe_layer* layer, int64_t M, int32_t top_k) {
  return qmoe_workspace_size_ex(layer, M, top_k, nullptr);
}

qmoe_status qmoe_forward_ex(const qmoe_layer* layer, const void* x, int64_t M, const int32_t* topk_ids,
                            const float* topk_weights, int32_t top_k, void* out, void* workspace,
                            size_t workspace_bytes, void* stream, const qmoe_options* opts) {
  return forward_impl(layer, x, M, topk_ids, topk_weights, top_k, out, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), opts);
}

qmoe_status qmoe_forward(const qmoe_layer* layer, const void* x, int64_t M, const int32_t* topk_ids,
                         const float* topk_weights, int32_t top_k, void* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return forward_impl(layer, x, M, topk_ids, topk_weights, top_k, out, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), nullptr);
}

qmoe_status qmoe_forward_profiled(const qmoe_layer* layer, const void* x, int64_t M, const int32_t* topk_ids,
                                  const float* topk_weights, int32_t top_k, void* out, void* workspace,
                                  size_t workspace_bytes, void* stream, const qmoe_options* opts,
                                  void* const* events, int32_t n_events, int32_t* n_launches) {
  if (events == nullptr || n_events < 14) return QMOE_ERR_INVALID_ARG;
  for (int i = 0; i < 14; ++i)
    if (events[i] == nullptr) return QMOE_ERR_INVALID_ARG;
  if (n_launches != nullptr) *n_launches = 0;
  return forward_impl(layer, x, M, topk_ids, topk_weights, top_k, out, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), opts, events, n_launches);
}

size_t qmoe_workspace_size_host(const qmoe_layer* layer, int64_t M, int32_t top_k) {
  const size_t w = qmoe_workspace_size(layer, M, top_k);
  if (w == 0) return 0;
  return al256(w) + host_staging_bytes(layer, M, top_k);
}

qmoe_status qmoe_forward_host(const qmoe_layer* layer, const void* x_host, int64_t M, const int32_t* topk_ids_host,
                              const float* topk_weights_host, int32_t top_k, void* out_host, void* workspace,
                              size_t workspace_bytes, void* stream) {
  const size_t w = qmoe_workspace_size(layer, M, top_k);
  if (w == 0) return validate_layer_dims(layer) != QMOE_OK ? validate_layer_dims(layer) : QMOE_ERR_INVALID_ARG;
  if (M == 0) return QMOE_OK;
  if (!x_host || !topk_ids_host || !topk_weights_host || !out_host) return QMOE_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < qmoe_workspace_size_host(layer, M, top_k)) return QMOE_ERR_WORKSPACE;
  const size_t xb = static_cast<size_t>(M) * layer->H * 2;
  const size_t pb = static_cast<size_t>(M) * top_k * 4;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Page-locked host buffers that the GPU can address (over NVLink-C2C on a
  // Grace-Blackwell node): the forward reads the inputs and writes the output
  // in place, with no staging copies; other host memory is staged below.
  const void* xm = mapped_host_ptr(x_host);
  const void* im = mapped_host_ptr(topk_ids_host);
  const void* wm = mapped_host_ptr(topk_weights_host);
  const void* om = mapped_host_ptr(out_host);
  if (xm != nullptr && im != nullptr && wm != nullptr && om != nullptr && aligned(xm, 256) && aligned(om, 256) &&
      aligned(im, 4) && aligned(wm, 4))
    return forward_impl(layer, xm, M, static_cast<const int32_t*>(im), static_cast<const float*>(wm), top_k,
                        const_cast<void*>(om), workspace, w, s, nullptr, nullptr, nullptr, true);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* stage = base + al256(w);
  void* x_dev = stage;
  int32_t* ids_dev = reinterpret_cast<int32_t*>(stage + al256(xb));
  float* w_dev = reinterpret_cast<float*>(stage + al256(xb) + al256(pb));
  void* out_dev = stage + al256(xb) + 2 * al256(pb);
  if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(ids_dev, topk_ids_host, pb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(w_dev, topk_weights_host, pb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  const qmoe_status st = forward_impl(layer, x_dev, M, ids_dev, w_dev, top_k, out_dev, workspace, w, s, nullptr);
  if (st != QMOE_OK) return st;
  if (cudaMemcpyAsync(out_host, out_dev, xb, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  return QMOE_OK;
}

qmoe_status qmoe_route_topk(const void* logits, qmoe_dtype logits_dtype, int64_t M, int32_t E, int32_t top_k,
                            int32_t renormalize, int32_t* topk_ids, float* topk_weights, void* stream) {
  if (M < 0 || E < 1 || E > 1024 || top_k < 1 || top_k > E) return QMOE_ERR_INVALID_ARG;
  if (top_k > 32) return QMOE_ERR_UNSUPPORTED;
  int dt = 0;
  if (logits_dtype == QMOE_F32)
    dt = 0;
  else if (logits_dtype == QMOE_F16)
    dt = 1;
  else if (logits_dtype == QMOE_BF16)
    dt = 2;
  else
    return QMOE_ERR_INVALID_ARG;
  if (M == 0) return QMOE_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  qmoe_status st;
  const void* ptrs[] = {logits, topk_ids, topk_weights};
  for (const void* p : ptrs)
    if ((st = check_dev_ptr(p, dev)) != QMOE_OK) return st;
  if (!aligned(logits, dt == 0 ? 4 : 2) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4))
    return QMOE_ERR_INVALID_ARG;
  const cudaError_t err = launch_route_topk(logits, dt, M, E, top_k, renormalize != 0 ? 1 : 0, topk_ids,
                                            topk_weights, current_sm_count(), static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

size_t qmoe_workspace_size_logits(const qmoe_layer* layer, int64_t M, int32_t top_k) {
  const size_t w = qmoe_workspace_size(layer, M, top_k);
  if (w == 0) return 0;
  return al256(w) + 2 * al256(static_cast<size_t>(M) * top_k * 4);
}

qmoe_status qmoe_forward_logits(const qmoe_layer* layer, const void* x, int64_t M, const void* logits,
                                qmoe_dtype logits_dtype, int32_t top_k, int32_t renormalize, void* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  const size_t w = qmoe_workspace_size(layer, M, top_k);
  if (w == 0) return validate_layer_dims(layer) != QMOE_OK ? validate_layer_dims(layer) : QMOE_ERR_INVALID_ARG;
  if (M == 0) return QMOE_OK;
  if (workspace == nullptr || workspace_bytes < qmoe_workspace_size_logits(layer, M, top_k)) return QMOE_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int32_t* ids = reinterpret_cast<int32_t*>(base + al256(w));
  float* wts = reinterpret_cast<float*>(base + al256(w) + al256(static_cast<size_t>(M) * top_k * 4));
  qmoe_status st = qmoe_route_topk(logits, logits_dtype, M, layer->E, top_k, renormalize, ids, wts, stream);
  if (st != QMOE_OK) return st;
  return forward_impl(layer, x, M, ids, wts, top_k, out, workspace, w, static_cast<cudaStream_t>(stream), nullptr);
}

qmoe_status qmoe_pack_int8_24(int32_t E, int32_t H, int32_t I, int32_t group_size, qmoe_dtype scale_dtype,
                              const int8_t* q13, const void* s13, const int8_t* q2, const void* s2, void* w13_packed,
                              float* s13_packed, void* w2_packed, float* s2_packed) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  const bool cw = group_size == -1;
  if (cw ? scale_dtype != QMOE_F32 : (scale_dtype != QMOE_F16 && scale_dtype != QMOE_BF16)) return QMOE_ERR_UNSUPPORTED;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed || (cw && (!s13_packed || !s2_packed)))
    return QMOE_ERR_INVALID_ARG;
  std::atomic<bool> bad{false};
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_24, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_24, 1, H, I, group_size);
  const uint16_t* g13 = cw ? nullptr : static_cast<const uint16_t*>(s13);
  const uint16_t* g2 = cw ? nullptr : static_cast<const uint16_t*>(s2);
  parallel_for(E, [&](int64_t e) {
    pack_int8_24_matrix(q13 + static_cast<size_t>(e) * 2 * I * H, g13 ? g13 + static_cast<size_t>(e) * (H / 128) * 2 * I : nullptr,
                        2 * I, H, I, static_cast<uint8_t*>(w13_packed) + e * b13, bad);
    pack_int8_24_matrix(q2 + static_cast<size_t>(e) * H * I, g2 ? g2 + static_cast<size_t>(e) * (I / 128) * H : nullptr, H,
                        I, 0, static_cast<uint8_t*>(w2_packed) + e * b2, bad);
    if (cw) {
      const float* f13 = static_cast<const float*>(s13);
      for (int t = 0; t < 2 * I / 128; ++t)
        for (int r = 0; r < 128; ++r)
          s13_packed[static_cast<size_t>(e) * 2 * I + t * 128 + r] = f13[static_cast<size_t>(e) * 2 * I + w13_canon_row(t, r, I, nullptr)];
      std::memcpy(s2_packed + static_cast<size_t>(e) * H, static_cast<const float*>(s2) + static_cast<size_t>(e) * H,
                  sizeof(float) * H);
    }
  });
  return bad ? QMOE_ERR_INVALID_ARG : QMOE_OK;
}

qmoe_status qmoe_unpack_int8_24(int32_t E, int32_t H, int32_t I, int32_t group_size, const void* w13_packed,
                                const float* s13_packed, const void* w2_packed, const float* s2_packed, int8_t* q13,
                                void* s13, int8_t* q2, void* s2) {
  if (!pack_dims_ok(E, H, I)) return QMOE_ERR_INVALID_ARG;
  if (group_size != 128 && group_size != -1) return QMOE_ERR_UNSUPPORTED;
  const bool cw = group_size == -1;
  if (!q13 || !s13 || !q2 || !s2 || !w13_packed || !w2_packed || (cw && (!s13_packed || !s2_packed)))
    return QMOE_ERR_INVALID_ARG;
  const size_t b13 = qmoe_packed_bytes(QMOE_INT8_24, 1, 2 * I, H, group_size);
  const size_t b2 = qmoe_packed_bytes(QMOE_INT8_24, 1, H, I, group_size);
  parallel_for(E, [&](int64_t e) {
    unpack_int8_24_matrix(static_cast<const uint8_t*>(w13_packed) + e * b13, !cw, 2 * I, H, I,
                          q13 + static_cast<size_t>(e) * 2 * I * H,
                          cw ? nullptr : static_cast<uint16_t*>(s13) + static_cast<size_t>(e) * (H / 128) * 2 * I);
    unpack_int8_24_matrix(static_cast<const uint8_t*>(w2_packed) + e * b2, !cw, H, I, 0,
                          q2 + static_cast<size_t>(e) * H * I,
                          cw ? nullptr : static_cast<uint16_t*>(s2) + static_cast<size_t>(e) * (I / 128) * H);
    if (cw) {
      float* f13 = static_cast<float*>(s13);
      for (int t = 0; t < 2 * I / 128; ++t)
        for (int r = 0; r < 128; ++r)
          f13[static_cast<size_t>(e) * 2 * I + w13_canon_row(t, r, I, nullptr)] = s13_packed[static_cast<size_t>(e) * 2 * I + t * 128 + r];
      std::memcpy(static_cast<float*>(s2) + static_cast<size_t>(e) * H, s2_packed + static_cast<size_t>(e) * H,
                  sizeof(float) * H);
    }
  });
  return QMOE_OK;
}

qmoe_status qmoe_pack_linear(qmoe_quant_type qt, int32_t N, int32_t K, int32_t group_size, qmoe_dtype scale_dtype,
                             const void* q, const void* s, const uint8_t* z, const int32_t* g_idx, void* w_packed,
                             float* s_packed, int32_t* perm_out) {
  if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return QMOE_ERR_INVALID_ARG;
  if (qmoe_packed_bytes(qt, 1, N, K, group_size) == 0) return QMOE_ERR_UNSUPPORTED;
  if (!q || !s || !w_packed) return QMOE_ERR_INVALID_ARG;
  const bool act_ok = scale_dtype == QMOE_F16 || scale_dtype == QMOE_BF16;
  const bool row_scales = has_row_scales(qt, group_size);
  if (row_scales ? scale_dtype != QMOE_F32 : !act_ok) return QMOE_ERR_UNSUPPORTED;
  if (row_scales && !s_packed) return QMOE_ERR_INVALID_ARG;
  if ((z != nullptr) != (qt == QMOE_INT4_GROUP_ZP)) return QMOE_ERR_INVALID_ARG;
  const bool int4_any = qt == QMOE_INT4_GROUP || qt == QMOE_INT4_GROUP_ZP;
  if (g_idx && (!int4_any || group_size != 128)) return QMOE_ERR_UNSUPPORTED;
  if (g_idx && !perm_out) return QMOE_ERR_INVALID_ARG;
  std::atomic<bool> bad{false};
  std::vector<int32_t> perm;
  if (g_idx) {
    if (!sorted_by_group(g_idx, K, perm)) return QMOE_ERR_UNSUPPORTED;
    std::memcpy(perm_out, perm.data(), sizeof(int32_t) * K);
  }
  uint8_t* out = static_cast<uint8_t*>(w_packed);
  const bool cw = group_size == -1;
  switch (qt) {
    case QMOE_INT4_GROUP:
    case QMOE_INT4_GROUP_ZP:
      pack_int4_matrix(static_cast<const uint8_t*>(q), static_cast<const uint16_t*>(s), z, cw, N, K, 0, nullptr,
                       g_idx ? perm.data() : nullptr, out, bad);
      break;
    case QMOE_INT4_GROUP_24:
      pack_int4_24_matrix(static_cast<const uint8_t*>(q), static_cast<const uint16_t*>(s), cw, N, K, 0, out, bad);
      break;
    case QMOE_INT8_GROUP:
      pack_int8_matrix(static_cast<const int8_t*>(q), static_cast<const uint16_t*>(s), N, K, 0, out, bad);
      break;
    case QMOE_INT8_24:
      pack_int8_24_matrix(static_cast<const int8_t*>(q), cw ? nullptr : static_cast<const uint16_t*>(s), N, K, 0, out,
                          bad);
      break;
    default:
      pack_int8_matrix(static_cast<const int8_t*>(q), nullptr, N, K, 0, out, bad);
      break;
  }
  if (row_scales) std::memcpy(s_packed, s, sizeof(float) * N);
  return bad ? QMOE_ERR_INVALID_ARG : QMOE_OK;
}

qmoe_status qmoe_unpack_linear(qmoe_quant_type qt, int32_t N, int32_t K, int32_t group_size, const void* w_packed,
                               const float* s_packed, const int32_t* g_idx, void* q, void* s, uint8_t* z) {
  if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return QMOE_ERR_INVALID_ARG;
  if (qmoe_packed_bytes(qt, 1, N, K, group_size) == 0) return QMOE_ERR_UNSUPPORTED;
  const bool row_scales = has_row_scales(qt, group_size);
  if (!w_packed || !q || !s || (row_scales && !s_packed) || ((z != nullptr) != (qt == QMOE_INT4_GROUP_ZP)))
    return QMOE_ERR_INVALID_ARG;
  std::vector<int32_t> perm;
  if (g_idx && !sorted_by_group(g_idx, K, perm)) return QMOE_ERR_UNSUPPORTED;
  const uint8_t* in = static_cast<const uint8_t*>(w_packed);
  const bool cw = group_size == -1;
  switch (qt) {
    case QMOE_INT4_GROUP:
    case QMOE_INT4_GROUP_ZP:
      unpack_int4_matrix(in, z != nullptr, cw, N, K, 0, nullptr, g_idx ? perm.data() : nullptr,
                         static_cast<uint8_t*>(q), static_cast<uint16_t*>(s), z);
      break;
    case QMOE_INT4_GROUP_24:
      unpack_int4_24_matrix(in, cw, N, K, 0, static_cast<uint8_t*>(q), static_cast<uint16_t*>(s));
      break;
    case QMOE_INT8_GROUP:
      unpack_int8_matrix(in, true, N, K, 0, static_cast<int8_t*>(q), static_cast<uint16_t*>(s));
      break;
    case QMOE_INT8_24:
      unpack_int8_24_matrix(in, !cw, N, K, 0, static_cast<int8_t*>(q), cw ? nullptr : static_cast<uint16_t*>(s));
      break;
    default:
      unpack_int8_matrix(in, false, N, K, 0, static_cast<int8_t*>(q), nullptr);
      break;
  }
  if (row_scales) std::memcpy(s, s_packed, sizeof(float) * N);
  return QMOE_OK;
}

size_t qmoe_linear_workspace_size(const qmoe_linear* layer, int64_t M, const qmoe_options* opts) {
  LinearPlan lp;
  if (make_linear_plan(layer, M, opts, current_sm_count(), &lp) != QMOE_OK) return 0;
  return lp.total;
}

qmoe_status qmoe_linear_describe_plan(const qmoe_linear* layer, int64_t M, const qmoe_options* opts, int32_t num_sms,
                                      qmoe_plan_info* info) {
  if (info == nullptr || num_sms < 0) return QMOE_ERR_INVALID_ARG;
  LinearPlan lp;
  const qmoe_status st = make_linear_plan(layer, M, opts, num_sms > 0 ? num_sms : current_sm_count(), &lp);
  if (st != QMOE_OK) return st;
  *info = qmoe_plan_info{};
  info->token_tile = lp.g.T;
  info->issuers = lp.g.issuers;
  info->acc_bufs = lp.g.acc_bufs;
  info->split1 = lp.g.S1;
  info->split2 = 0;
  info->w_stages = lp.g.w_stages;
  info->ab_stages = lp.g.ab_stages;
  info->b_stages = lp.g.b_stages;
  info->dq_sets = lp.g.dq_sets;
  info->cta_pair = 0;
  info->cta_pair_down = 0;
  info->stage_bytes = lp.g.stage_bytes;
  info->workspace_bytes = static_cast<int64_t>(lp.total);
  return QMOE_OK;
}

qmoe_status qmoe_linear_forward(const qmoe_linear* layer, const void* x, int64_t M, void* out, void* workspace,
                                size_t workspace_bytes, void* stream, const qmoe_options* opts) {
  return linear_forward_impl(layer, x, M, out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), opts);
}

qmoe_status qmoe_read_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return QMOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return QMOE_ERR_CUDA;
  }
  return static_cast<qmoe_status>(v);
}

}  // extern "C"
