// prefill.cu -- chunked prefill over 16-token pages on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Method (what is computed): chunk row i of sequence b sits at position
// p = past_b + i and attends over keys j <= p with p - j < W (all j <= p for a
// full layer): the band rule "key j hidden from query i when past + i - j >= W"
// composed with the aligned causal rule (InfiniLM PR 581 "feat: support gemma2
// and gemma3_text", Gemma-3 item 3), scores s = scale * q.k with the optional
// softcap cap * tanh(s / cap) before the softmax (same PR, Gemma-2 item 1),
// GQA query heads of one KV head folded into the rows of a tile (same item's
// head-major repacking), keys and values gathered through the block table
// ("Gemma 4 model architecture analysis", sections 6.3 and 6.5); the key range
// of a tile is cut to what the band leaves visible (the PR's follow-up item 2).
//
// Design (how, on sm_103a):
//  * Work item = (sequence, block of 128/G chunk tokens, KV head, half of
//    head_dim for head_dim 512): 128 query rows = (128/G tokens) x (G heads),
//    token-major. A plan kernel lists the (sequence, block) units sorted by
//    their number of key tiles, longest first; a persistent grid of one CTA
//    per SM takes items from that list with an atomic counter, so long items
//    start first and short ones fill the gaps (longest-processing-time order).
//  * Each CTA runs warp-specialised pipelines that carry on across items:
//    warp 8 takes the next item, loads Q (TMA, 128-byte swizzle) and streams
//    K tiles of BN keys (64, or 32 at head_dim 512 without k_eq_v) into a
//    ring, one TMA box per 8 keys over the whole head, or over one head_dim
//    half at head_dim 512 with k_eq_v ([group][chunk][8 rows][128 B], so the
//    8-row groups of the K-major operand sit a fixed stride apart); warp 10
//    streams V tiles into a second ring. A K stage is released once QK has
//    read it (with k_eq_v: the stage holding V after PV), a V stage after PV.
//  * Two warps issue tcgen05.mma (one elected thread each): warp 9 the QK
//    stream S_j = Q K_j^T (SS, both K-major) into one of four S/P buffers in
//    tensor memory, warp 11 the PV stream O += P_j V_j (TS: P from the same
//    buffer, where the softmax wrote it over S_j; V MN-major). QK runs up to
//    four tiles ahead of PV, so S is ready whenever the softmax is; the next
//    item's QK starts as soon as its Q has landed, while the softmax warps
//    still finish the previous item.
//  * Warps 0-3 run the softmax: warp w owns the 32 rows of tensor-memory lane
//    quadrant w and all key columns of a tile, so row maxima and sums stay in
//    one thread and the softmax warps never wait for each other. The row
//    maximum comes from the raw scores (the softcap is monotone); the softcap
//    is an odd polynomial on the FMA pipe where every |s/cap| of the warp's
//    tile is at most 1/4 (the exp formula elsewhere); the band/causal
//    predicate is applied on edge tiles only; the online softmax runs in fp32
//    in the exp2 domain with a running maximum first set a factor 2^64
//    above the largest score seen and raised (O rescaled) only when a score
//    exceeds it by another 2^64 (rescales are rare). P is written back to tensor
//    memory as a bf16 high part and a bf16 remainder (integer ops); both
//    are multiplied into O, so P enters the product to 2^-14 relative.
//  * Warps 4-7 are the epilogue: once an item's last PV is done they scale
//    its O by 1/l, stage it per warp through shared memory 32 columns at a
//    time and write whole 128-byte row segments, while the softmax warps
//    already work on the next item.
//  * V rows of key positions that no row of the item can see (before the
//    window of its first row, after its last row) are zeroed in shared memory
//    so uncached or stale slots never reach O.
//  * Every wait is bounded; on timeout the kernel flags PSW_DEVERR_PIPELINE,
//    every role leaves its loop, drains its own copies and MMAs, and the
//    tensor memory is freed before the CTA exits.
#include <math.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace pf {

constexpr int kSoftmaxWarps = 4;  // warps 0-3
constexpr int kEpiWarps = 4;      // warps 4-7
constexpr int kKWarp = 8;    // takes work items, loads Q and K tiles
constexpr int kQkWarp = 9;   // tcgen05.mma issuer of the QK stream
constexpr int kVWarp = 10;   // V tiles (idle with k_eq_v)
constexpr int kPvWarp = 11;  // tcgen05.mma issuer of the PV stream
constexpr int kThreads = 12 * 32;
constexpr int kRows = 128;
constexpr int kPageBoxBytes = kBlockSize * 128;  // one TMA box: 16 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Running maximum m of a row (log2 units). When a row's first visible keys
// arrive, m is set kMaxBias above their largest score; afterwards it is raised
// (and O rescaled by 2^(m_old - m_new)) only once a score exceeds it by more
// than kRescaleThreshold, and then to that score. So P = 2^(z - m) <= 2^64,
// l < 2^95 for up to 2^31 keys and O stays below the fp32 limit while
// |V| < 2^33. Keys more than 62 below the row's first maximum flush to zero
// (below 2^-62 of that key). The rescale factor underflows only when the old
// terms, at most 2^64 before it, fall below 2^-62 of the new maximum key.
// Rescales of O wait for the previous PV, so they should be rare: a row's
// maximum must grow by 128 after its first visible keys (a row whose first
// tile holds few of its keys would otherwise rescale on its second tile,
// while the accumulator may still be held by the previous item's epilogue).
constexpr float kRescaleThreshold = 64.f;
constexpr float kMaxBias = 64.f;
constexpr int kCostBuckets = 4096;       // plan: units sorted by tile count (capped)
constexpr int kPlanThreads = 1024;

// Work list at the start of the workspace: this header, then int2 units.
struct PlanHeader {
  int32_t next_item;  // atomic work counter
  int32_t n_units;    // (sequence, block) units in the list
  int32_t pad[14];
};
static_assert(sizeof(PlanHeader) == 64, "plan header");

template <int HD, bool KEQV>
struct Cfg {
  static constexpr int kQChunks = HD / 64;
  // head_dim 512 with k_eq_v: 64-key tiles loaded as two stages of one
  // head_dim half each, the half that is not this item's V first; it is
  // released once QK has read it, the item's own half (its V) after PV. The
  // 128 KB Q tile is then read by the QK MMAs once per 64 keys, not per 32.
  static constexpr bool kSplitK = (HD == 512) && KEQV;
  static constexpr int kKHalves = kSplitK ? 2 : 1;  // K stages per tile
  static constexpr int kBN = (HD == 256 || kSplitK) ? 64 : 32;
  static constexpr int kPagesPerTile = kBN / kBlockSize;
  static constexpr int kOCols = 256;
  static constexpr int kDSplit = HD / kOCols;
  static constexpr int kVChunks = kOCols / 64;
  static constexpr int kQBytes = kQChunks * kRows * 128;
  static constexpr int kChunkTileBytes = kBN * 128;  // one 64-column chunk of a K/V tile
  // K stage: [8-key group][chunk][8 rows][128 B], one TMA box per group (all
  // chunks of the head, or the chunks of one head_dim half with kSplitK)
  static constexpr int kKBoxChunks = kQChunks / kKHalves;
  static constexpr int kKGroupBytes = kKBoxChunks * 1024;
  static constexpr int kKBoxes = kBN / 8;
  static constexpr int kKBytes = kKBoxes * kKGroupBytes;
  static constexpr int kVBytes = KEQV ? 0 : kVChunks * kChunkTileBytes;
  static constexpr int kVPageBytes = kVChunks * kPageBoxBytes;  // one page of V
  static constexpr int kBarsBytes = 2432;
  static constexpr int kAvail = 232448 - kBarsBytes;
  static constexpr int kRingBudget = kAvail - kQBytes;
  static constexpr int kVStages = KEQV ? 0 : 2;
  static constexpr int kKStagesFit = (kRingBudget - kVStages * kVBytes) / kKBytes;
  static constexpr int kKStages = kKStagesFit > 4 ? 4 : kKStagesFit;
  static constexpr int kVS = kVStages > 0 ? kVStages : 1;  // ring size for index math
  static constexpr int kUsed =
      kQBytes + kKStages * kKBytes + kVStages * kVBytes + kBarsBytes;
  // slack to round the dynamic shared memory base up to 1024 bytes (128-byte
  // swizzle atoms); checked at run time
  static constexpr int kSlack = (232448 - kUsed) < 1024 ? (232448 - kUsed) : 1024;
  static constexpr int kSmemBytes = kUsed + kSlack;
  // tensor memory columns: O | four S/P buffers
  static constexpr int kTmemO = 0;
  // S/P buffers: S_g lands in buffer g mod kSP; the softmax reads all of it
  // and writes P_g (bf16 hi in the first kBN/2 columns, lo in the next) over it
  static constexpr int kSP = 4;
  static constexpr int kTmemS = 256;  // + b * kBN
  static constexpr int kTmemCols = 512;
  static_assert(kKStages >= 2 * kKHalves - (kSplitK ? 1 : 0), "K stages");
  static_assert(kKBoxes <= 32 && kPagesPerTile <= 32,
                "one TMA box per producer lane");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kTmemS + kSP * kBN <= kTmemCols, "tensor memory columns");
};

struct Bars {
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[2], v_empty[2];
  uint64_t s_full[4], p_full[4], p_free[4];
  uint64_t o_full, o_free;
  uint64_t mma_drained;
  uint64_t v_fix;  // a V tile with hidden rows lands here before they are zeroed
  int32_t item[2];
  uint32_t tmem_base;
  int32_t abort;
  uint64_t stats_full[2], stats_free[2];  // row maxima and sums, per item parity
  float stat_m[2][kRows], stat_l[2][kRows];
};

// Geometry of one (sequence, block) unit; uniform across a CTA.
struct Geom {
  int b, q0, past, i0, tok_valid;
  int j_lo, j_hi;  // keys [j_lo, j_hi] are visible to some row of the block
  int kt0, nkt;    // key tiles kt0 .. kt0 + nkt - 1
  int last_page;   // last page index that may be read
};

// Returns false when the block has no rows. With `err`, length and capacity
// problems are reported (once per sequence: by its first block).
__device__ __forceinline__ bool unit_geom(int b, int rb, const int32_t* __restrict__ cu_q,
                                          const int32_t* __restrict__ past_lens, int n_q_total,
                                          int max_q_len, int max_blocks, int window, int T, int BN,
                                          Geom& g, int32_t* err) {
  const int q0 = cu_q[b];
  int n_b = cu_q[b + 1] - q0;
  const int past = past_lens[b];
  // positions must stay far from int overflow (past + rows + one tile)
  if (n_b < 0 || past < 0 || q0 < 0 ||
      static_cast<int64_t>(past) + max_q_len > 0x7fffffffLL - 4096) {
    if (err != nullptr && rb == 0) flag_error(err, PSW_DEVERR_LENGTH);
    return false;
  }
  if (n_b > max_q_len || static_cast<int64_t>(q0) + n_b > n_q_total) {
    if (err != nullptr && rb == 0) flag_error(err, PSW_DEVERR_LENGTH);
    n_b = min(max_q_len, n_q_total - q0);
  }
  const int i0 = rb * T;
  if (i0 >= n_b) return false;
  g.b = b;
  g.q0 = q0;
  g.past = past;
  g.i0 = i0;
  g.tok_valid = min(T, n_b - i0);
  const int p_lo = past + i0;
  const int p_hi = past + i0 + g.tok_valid - 1;
  const int seq_end = past + n_b;  // positions < seq_end are cached
  if (err != nullptr && rb == 0 &&
      static_cast<int64_t>(seq_end) > static_cast<int64_t>(max_blocks) * kBlockSize)
    flag_error(err, PSW_DEVERR_CAPACITY);
  g.j_lo = (window > 0) ? max(0, p_lo - window + 1) : 0;
  g.j_hi = p_hi;
  g.kt0 = g.j_lo / BN;
  g.nkt = g.j_hi / BN - g.kt0 + 1;
  g.last_page = min((seq_end - 1) / kBlockSize, max_blocks - 1);
  return true;
}

// ---------------------------------------------------------------- plan
// One CTA: counts the key tiles of every (sequence, block) unit, orders the
// units by that count, longest first (a counting sort over kCostBuckets
// buckets; counts beyond the last bucket share it), and resets the work
// counter of the main kernel. Length and capacity errors are reported here.
__global__ void __launch_bounds__(kPlanThreads)
prefill_plan_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ past_lens,
                    int n_seqs, int n_q_total, int max_q_len, int max_blocks, int window, int T,
                    int BN, int max_rb, PlanHeader* hdr, int2* __restrict__ units,
                    int32_t* err) {
  __shared__ int cnt[kCostBuckets];
  __shared__ int warp_tot[kPlanThreads / 32];
  constexpr int kPer = kCostBuckets / kPlanThreads;  // buckets per thread
  const int tid = threadIdx.x;
  for (int i = tid; i < kCostBuckets; i += kPlanThreads) cnt[i] = 0;
  __syncthreads();
  const int64_t n_pot = static_cast<int64_t>(n_seqs) * max_rb;
  for (int64_t u = tid; u < n_pot; u += kPlanThreads) {
    const int b = static_cast<int>(u / max_rb);
    const int rb = static_cast<int>(u - static_cast<int64_t>(b) * max_rb);
    Geom g;
    if (!unit_geom(b, rb, cu_q, past_lens, n_q_total, max_q_len, max_blocks, window, T, BN, g,
                   err))
      continue;
    atomicAdd(&cnt[min(g.nkt, kCostBuckets - 1)], 1);
  }
  __syncthreads();
  // Descending bucket order: thread t owns buckets kCostBuckets-1-kPer*t and
  // the kPer - 1 below it; an exclusive scan of the per-thread sums gives the
  // first list slot of every bucket.
  int local[kPer];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    local[i] = cnt[kCostBuckets - 1 - (kPer * tid + i)];
    sum += local[i];
  }
  const int lane = tid & 31, wid = tid >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix over warps
  }
  __syncthreads();
  int base = warp_tot[wid] + incl - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    cnt[kCostBuckets - 1 - (kPer * tid + i)] = base;  // first slot of this bucket
    base += local[i];
  }
  if (tid == kPlanThreads - 1) hdr->n_units = base;  // the last thread ends at the total
  __syncthreads();
  for (int64_t u = tid; u < n_pot; u += kPlanThreads) {
    const int b = static_cast<int>(u / max_rb);
    const int rb = static_cast<int>(u - static_cast<int64_t>(b) * max_rb);
    Geom g;
    if (!unit_geom(b, rb, cu_q, past_lens, n_q_total, max_q_len, max_blocks, window, T, BN, g,
                   nullptr))
      continue;
    const int pos = atomicAdd(&cnt[min(g.nkt, kCostBuckets - 1)], 1);
    units[pos] = make_int2(b, rb);
  }
  if (tid == 0) hdr->next_item = 0;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from shared to global memory, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk copy of this thread has read its source.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ---------------------------------------------------------------- softcap
// tanh(y) for |y| <= 1/4: the odd Taylor polynomial through y^7; the first
// omitted term, 62/2835 y^9, is below 8.3e-8 there.
__device__ __forceinline__ float tanh_p7(float y) {
  const float y2 = y * y;
  const float r = fmaf(fmaf(-17.f / 315.f, y2, 2.f / 15.f), y2, -1.f / 3.f);
  return fmaf(r * y2, y, y);
}

// z = x (A + x^2 (C1 + x^2 (C2 + x^2 C3))) + c0 on N raw scores x, two per
// packed register, in Horner form (without softcap C1 = C2 = C3 = 0 and only
// A x + c0 is formed): five packed FMAs per pair. Every Horner step runs over
// 16 pairs before the next, so the dependent FMAs of one pair interleave with
// those of the others.
template <int N>
__device__ __forceinline__ void log2_terms(const float* x, uint64_t* z2, bool cap, float A,
                                           float C1, float C2, float C3, float c0) {
  constexpr int G = (N / 2 < 16) ? N / 2 : 16;
  const uint64_t A2 = f2_pack(A, A), c02 = f2_pack(c0, c0);
  const uint64_t C12 = f2_pack(C1, C1), C22 = f2_pack(C2, C2), C32 = f2_pack(C3, C3);
#pragma unroll
  for (int gb = 0; gb < N / 2; gb += G) {
    uint64_t xx[G];
#pragma unroll
    for (int k = 0; k < G; ++k) xx[k] = f2_pack(x[2 * (gb + k)], x[2 * (gb + k) + 1]);
    if (cap) {
      uint64_t xq[G], r[G];
#pragma unroll
      for (int k = 0; k < G; ++k) xq[k] = f2_mul(xx[k], xx[k]);
#pragma unroll
      for (int k = 0; k < G; ++k) r[k] = f2_fma(C32, xq[k], C22);
#pragma unroll
      for (int k = 0; k < G; ++k) r[k] = f2_fma(r[k], xq[k], C12);
#pragma unroll
      for (int k = 0; k < G; ++k) r[k] = f2_fma(r[k], xq[k], A2);
#pragma unroll
      for (int k = 0; k < G; ++k) z2[gb + k] = f2_fma(xx[k], r[k], c02);
    } else {
#pragma unroll
      for (int k = 0; k < G; ++k) z2[gb + k] = f2_fma(xx[k], A2, c02);
    }
  }
}

// tanh(y) for any y as 1 - 2 / (e^{2|y|} + 1) with the sign restored. Near 0
// its relative error grows, but its absolute error stays a few units in the
// last place of 1, and the softcap only needs the logit cap * tanh to absolute
// accuracy (P = exp(logit - max)).
__device__ __forceinline__ float tanh_exp(float y) {
  const float t = ex2_approx(-2.f * kLog2e * fabsf(y));  // e^{-2|y|}
  return copysignf(__fdividef(1.f - t, 1.f + t), y);
}

// maximum / minimum of N values (N a multiple of 8), four 3-input chains
template <int N>
__device__ __forceinline__ float max_of(const float* x) {
  float a = x[0], b = x[1], c = x[2], d = x[3];
#pragma unroll
  for (int i = 4; i + 7 < N + 4; i += 8) {
    a = max3f(a, x[i], x[i + 1]);
    b = max3f(b, x[i + 2], x[i + 3]);
    if (i + 7 < N) {
      c = max3f(c, x[i + 4], x[i + 5]);
      d = max3f(d, x[i + 6], x[i + 7]);
    }
  }
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}
template <int N>
__device__ __forceinline__ float min_of(const float* x) {
  float a = x[0], b = x[1], c = x[2], d = x[3];
#pragma unroll
  for (int i = 4; i + 7 < N + 4; i += 8) {
    a = min3f(a, x[i], x[i + 1]);
    b = min3f(b, x[i + 2], x[i + 3]);
    if (i + 7 < N) {
      c = min3f(c, x[i + 4], x[i + 5]);
      d = min3f(d, x[i + 6], x[i + 7]);
    }
  }
  return fminf(fminf(a, b), fminf(c, d));
}

// A whole warp waits for a phase: one non-blocking test first (the phase is
// usually complete already), the bounded blocking wait only when it is not.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// ---------------------------------------------------------------- kernel
template <int HD, bool KEQV>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
               const __grid_constant__ CUtensorMap v_map, const int32_t* __restrict__ cu_q,
               const int32_t* __restrict__ past_lens, const int32_t* __restrict__ block_table,
               int max_blocks, int64_t num_blocks, int n_q_total, int max_q_len, int n_q,
               int group, int window, float scale, float softcap, PlanHeader* hdr,
               const int2* __restrict__ units, float* __restrict__ out,
               float* __restrict__ lse, int32_t* err, int stall_cta, int stall_tile) {
  using C = Cfg<HD, KEQV>;
  constexpr int BN = C::kBN;
  constexpr int KS = C::kKStages;
  constexpr int VS = C::kVS;
  const int T = kRows / group;  // chunk tokens per item
  const int n_kv = n_q / group;
  const int subs = n_kv * C::kDSplit;  // items per unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(C::kSlack)) {  // uniform: every thread leaves
    if (threadIdx.x == 0) flag_error(err, PSW_DEVERR_PIPELINE);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* q_smem = smem;
  uint8_t* k_ring = smem + C::kQBytes;
  uint8_t* v_ring = k_ring + KS * C::kKBytes;
  Bars* bars = reinterpret_cast<Bars*>(v_ring + C::kVStages * C::kVBytes);
  static_assert(sizeof(Bars) <= C::kBarsBytes, "barrier block");

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->item_full[i], 1);
      // readers of an item id: the two MMA threads, the V producer, the
      // softmax and the epilogue warps
      mbar_init(&bars->item_empty[i], 2 + (KEQV ? 0 : 1) + kSoftmaxWarps + kEpiWarps);
      mbar_init(&bars->stats_full[i], kSoftmaxWarps);
      mbar_init(&bars->stats_free[i], kEpiWarps);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], kSoftmaxWarps);
      mbar_init(&bars->p_free[i], 1);
      mbar_init(&bars->s_full[i + 2], 1);
      mbar_init(&bars->p_full[i + 2], kSoftmaxWarps);
      mbar_init(&bars->p_free[i + 2], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_free, kEpiWarps);
    mbar_init(&bars->mma_drained, 2);  // one commit from each MMA thread
    mbar_init(&bars->v_fix, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tc::alloc(&bars->tmem_base, C::kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  const int n_items = hdr->n_units * subs;

  // item id -> KV head, head_dim half and geometry of its unit
  auto item_geom = [&](int item, int& kvh, int& dh, Geom& g) {
    const int u = item / subs;
    const int sub = item - u * subs;
    kvh = sub / C::kDSplit;
    dh = sub - kvh * C::kDSplit;
    const int2 unit = units[u];
    return unit_geom(unit.x, unit.y, cu_q, past_lens, n_q_total, max_q_len, max_blocks, window,
                     T, BN, g, nullptr);
  };

  if (warp == kKWarp || warp == kVWarp) {
    // ------------------------------------------------------------ producers
    const bool v_side = (warp == kVWarp);
    if (v_side && KEQV) goto done;  // V is the K tile
    if (!v_side && lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      if (!KEQV) prefetch_tensormap(&v_map);
    }
    constexpr int P = C::kPagesPerTile;
    constexpr int kTilesPerGroup = 32 / P;
    constexpr int kKBoxes = C::kKBoxes;
    const int k_lp = lane >> 1, k_half = lane & 1;  // K: half-page box of every chunk
    const int nst = v_side ? VS : KS;
    const int my_lp = v_side ? lane : k_lp;  // V: one whole-page box per lane
    int gt = 0;     // tiles issued by this warp over all items
    int nq = 0;     // Q tiles issued
    int n_fix = 0;  // V tiles that landed on v_fix
    bool ok = true;
    bool stalled = false;  // testing hook: the K copy gt == stall_tile is never issued
    for (int n = 0; ok; ++n) {
      // ---- the item: the K warp takes it and publishes it, the V warp reads it
      int item = -1;
      const int slot = n & 1;
      if (!v_side) {
        if (lane == 0) {
          if (n >= 2) ok = mbar_wait(&bars->item_empty[slot], ((n >> 1) - 1) & 1);
          if (ok) {
            const int it = *abort_flag ? n_items : atomicAdd(&hdr->next_item, 1);
            item = it < n_items ? it : -1;
            bars->item[slot] = item;
            mbar_arrive(&bars->item_full[slot]);
          }
        }
      } else {
        ok = mbar_wait(&bars->item_full[slot], (n >> 1) & 1);
        if (ok) item = bars->item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      item = __shfl_sync(0xffffffffu, item, 0);
      if (!ok || item < 0) break;
      int kvh, dh;
      Geom g;
      item_geom(item, kvh, dh, g);  // listed units always have rows
      // ---- Q, once the previous item no longer needs the Q tile (warmed in L2
      // first, so the load that waits for it finds it there)
      if (!v_side) {
        if (lane < C::kQChunks)
          tma_prefetch_3d(&q_map, lane * 64, kvh * group, g.q0 + g.i0);
        if (lane == 0) {
          if (nq > 0)
            ok = mbar_wait(&bars->q_empty, (nq - 1) & 1);
          if (ok && !*abort_flag) {
            mbar_arrive_expect_tx(&bars->q_full,
                                  static_cast<uint32_t>(C::kQChunks * group * T * 128));
            for (int c = 0; c < C::kQChunks; ++c)
              tma_load_3d(q_smem + c * (kRows * 128), &q_map, &bars->q_full, c * 64,
                          kvh * group, g.q0 + g.i0);
          } else {
            ok = false;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++nq;
      }
      // ---- K or V tiles. Block ids of the item's pages, 32 at a time: lane l
      // holds page first_page + 32 grp + l; the next group is read one ahead,
      // so a tile needs only shuffles.
      const int first_page = g.kt0 * P;
      const int32_t* bt_row = block_table + static_cast<int64_t>(g.b) * max_blocks;
      auto load_group = [&](int grp) -> int {
        const int page = first_page + grp * 32 + lane;
        if (grp * kTilesPerGroup >= g.nkt || page > g.last_page) return -1;
        int blk = bt_row[page];
        if (blk < 0 || blk >= num_blocks) {
          flag_error(err, PSW_DEVERR_BLOCK_ID);
          blk = -1;  // out-of-range box: TMA fills zeros
        }
        return blk;
      };
      int ids = load_group(0), ids_next = load_group(1);
      for (int j = 0; j < g.nkt && ok; ++j) {
        if (j > 0 && j % kTilesPerGroup == 0) {
          ids = ids_next;
          ids_next = load_group(j / kTilesPerGroup + 1);
        }
        const int src = (j % kTilesPerGroup) * P + (my_lp < P ? my_lp : 0);
        const int my_blk = __shfl_sync(0xffffffffu, ids, src);
        // V rows of keys that no row of the item may see (before the window
        // of its first row, after its last row) must not reach O: such a tile
        // lands on v_fix first, those rows are zeroed here, and only then is
        // v_full completed (by a plain arrival)
        const int key0 = (g.kt0 + j) * BN;
        const int z_lo = max(0, g.j_lo - key0);       // rows [0, z_lo) hidden
        const int z_hi = min(BN, g.j_hi - key0 + 1);  // rows [z_hi, BN) hidden
        const bool fix = v_side && (z_lo > 0 || z_hi < BN);
        const int n_st = v_side ? 1 : C::kKHalves;  // stages of this tile
        for (int hh = 0; hh < n_st; ++hh, ++gt) {
          const int stage = gt % nst;
          const uint32_t ph = static_cast<uint32_t>(gt / nst) & 1u;
          uint64_t* empty = v_side ? &bars->v_empty[stage] : &bars->k_empty[stage];
          uint64_t* full = v_side ? &bars->v_full[stage] : &bars->k_full[stage];
          if (!v_side && static_cast<int>(blockIdx.x) == stall_cta && gt == stall_tile) {
            stalled = true;  // leave quietly: the waits downstream must run out
            ok = false;
            break;
          }
          if (lane == 0) ok = mbar_wait(empty, ph ^ 1) && !*abort_flag;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane == 0)
            mbar_arrive_expect_tx(fix ? &bars->v_fix : full, v_side ? C::kVBytes : C::kKBytes);
          __syncwarp();
          if (!v_side) {
            // with kSplitK: head_dim half 1 - dh first (QK only), then half dh
            const int h = C::kSplitK ? (hh == 0 ? 1 - dh : dh) : 0;
            const int zc = kvh * C::kQChunks + h * C::kKBoxChunks;
            if (lane < kKBoxes) {
              tma_load_3d(k_ring + stage * C::kKBytes + lane * C::kKGroupBytes, &k_map, full, 0,
                          my_blk * kBlockSize + k_half * 8, zc);
            }
          } else {
            uint8_t* vt = v_ring + stage * C::kVBytes;
            if (lane < P) {  // V tile: [page][chunk][16 rows][128 B]
              const int z = kvh * C::kQChunks + dh * C::kVChunks;
              tma_load_3d(vt + lane * C::kVPageBytes, &v_map, fix ? &bars->v_fix : full, 0,
                          my_blk * kBlockSize, z);
            }
            if (fix) {
              if (lane == 0) ok = mbar_wait(&bars->v_fix, static_cast<uint32_t>(n_fix) & 1u);
              ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
              ++n_fix;
              if (!ok) break;
              for (int idx = lane; idx < BN * C::kVChunks * 8; idx += 32) {
                const int row = idx / (C::kVChunks * 8), rem = idx - row * (C::kVChunks * 8);
                const int cv = rem >> 3, u = rem & 7;
                if (row < z_lo || row >= z_hi)
                  *reinterpret_cast<uint4*>(vt + (row >> 4) * C::kVPageBytes +
                                            cv * kPageBoxBytes + (row & 15) * 128 + u * 16) =
                      make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();  // the tensor core reads these rows
              __syncwarp();
              if (lane == 0) mbar_arrive(full);
            }
          }
        }
      }
    }
    if (!ok && !stalled && lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *abort_flag = 1;
    }
    if (lane == 0) {  // drain this warp's own copies before anyone leaves
      if (!v_side && nq > 0) mbar_wait(&bars->q_full, (nq - 1) & 1);
      for (int i = max(0, gt - nst); i < gt; ++i)
        mbar_wait(v_side ? &bars->v_full[i % nst] : &bars->k_full[i % nst],
                  static_cast<uint32_t>(i / nst) & 1u);
    }
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ MMA issuers
    // Two warps issue tcgen05.mma, one elected thread each: warp kQkWarp the
    // QK stream S_g = Q K_g^T (into S/P buffer g mod 4, once PV has consumed
    // the P of tile g - 4 there and K_g has landed), warp kPvWarp the PV stream
    // O += P_g V_g (once P_g is in tensor memory and V_g has landed). Each
    // stream depends only on earlier tiles, a commit tracks only its own
    // thread's MMAs, and the tensor pipe interleaves the two streams.
    // Descriptors are a base plus compile-time offsets (the 14-bit address
    // field never carries: shared addresses stay below 2^18).
    const bool qk_side = (warp == kQkWarp);
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, BN, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, C::kOCols, 0, 1);
      const uint64_t q_desc = tc::smem_desc(smem_u32(q_smem), 16, 1024, tc::kSwizzle128B);
      const uint32_t k_base = smem_u32(k_ring);
      const uint32_t v_base = smem_u32(v_ring);
      bool ok = true;
      int g_tile = 0;
      for (int n = 0; ok; ++n) {
        ok = mbar_wait(&bars->item_full[n & 1], (n >> 1) & 1);
        if (!ok) break;
        const int item = bars->item[n & 1];
        mbar_arrive(&bars->item_empty[n & 1]);
        if (item < 0) break;
        int kvh, dh;
        Geom g;
        item_geom(item, kvh, dh, g);
        for (int j = 0; j < g.nkt && ok; ++j, ++g_tile) {
          const bool first = (j == 0), last = (j == g.nkt - 1);
          if (*abort_flag) {
            ok = false;
            break;
          }
          if (qk_side) {
            const int b = g_tile % C::kSP;  // its previous P (tile g - kSP) must be consumed
            ok = (!first || mbar_wait(&bars->q_full, n & 1)) &&
                 (g_tile < C::kSP ||
                  mbar_wait(&bars->p_free[b], ((g_tile / C::kSP) - 1) & 1));
            if (!ok) break;
            const uint32_t d = tmem + C::kTmemS + b * BN;
            constexpr int kSteps = HD / 16 / C::kKHalves;  // K16 steps per K stage
            constexpr int kQChunkBytes = kRows * 128;
#pragma unroll
            for (int hh = 0; hh < C::kKHalves; ++hh) {
              const int hc = g_tile * C::kKHalves + hh;  // K stage counter
              const int stage = hc % KS;
              ok = mbar_wait(&bars->k_full[stage], (hc / KS) & 1);
              if (!ok) break;
              tc::fence_after();
              // head_dim half held by this stage (kSplitK: 1 - dh, then dh)
              const int h = C::kSplitK ? (hh == 0 ? 1 - dh : dh) : 0;
              const uint64_t k_desc =
                  tc::smem_desc(k_base + stage * C::kKBytes, 16, C::kKGroupBytes, tc::kSwizzle128B);
#pragma unroll
              for (int kk = 0; kk < kSteps; ++kk) {
                const int ks = h * kSteps + kk;  // K16 step over head_dim
                const uint32_t off_q =
                    static_cast<uint32_t>((ks >> 2) * kQChunkBytes + (ks & 3) * 32) >> 4;
                const uint32_t off_k =
                    static_cast<uint32_t>((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
                tc::mma_ss(d, q_desc + off_q, k_desc + off_k, idesc_qk,
                           (hh > 0 || kk > 0) ? 1u : 0u);
              }
              // K read by QK (with kSplitK: the half that is not this item's V)
              if (!KEQV || (C::kSplitK && hh == 0)) tc::commit(&bars->k_empty[stage]);
            }
            if (!ok) break;
            tc::commit(&bars->s_full[b]);
            if (last) tc::commit(&bars->q_empty);  // the Q tile may be replaced
          } else {
            const int pb = g_tile % C::kSP;
            ok = mbar_wait(&bars->p_full[pb], (g_tile / C::kSP) & 1) &&
                 (KEQV || mbar_wait(&bars->v_full[g_tile % VS], (g_tile / VS) & 1)) &&
                 (!first || n == 0 || mbar_wait(&bars->o_free, (n - 1) & 1));
            if (!ok) break;
            tc::fence_after();
            // V with k_eq_v is the K tile ([8-key group][chunk][8 rows]); a V
            // tile of its own is [page][chunk][16 rows]; a K16 step is one page
            // (two 8-key groups) either way
            // with k_eq_v the K stage holding head_dim half dh (kSplitK: the
            // tile's second stage)
            const int vstage = (g_tile * C::kKHalves + C::kKHalves - 1) % KS;
            const uint32_t vb = KEQV ? k_base + vstage * C::kKBytes +
                                           (C::kSplitK ? 0 : dh * C::kVChunks * 1024)
                                     : v_base + (g_tile % VS) * C::kVBytes;
            const uint64_t v_desc =
                KEQV ? tc::smem_desc(vb, 1024, C::kKGroupBytes, tc::kSwizzle128B)
                     : tc::smem_desc(vb, kPageBoxBytes, 1024, tc::kSwizzle128B);
            constexpr int kPageStep = KEQV ? 2 * C::kKGroupBytes : C::kVPageBytes;
            const uint32_t p_hi = tmem + C::kTmemS + pb * BN;
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
              const uint64_t bdesc = v_desc + static_cast<uint32_t>((ks * kPageStep) >> 4);
              tc::mma_ts(tmem + C::kTmemO, p_hi + ks * 8, bdesc, idesc_pv,
                         (!first || ks > 0) ? 1u : 0u);
              tc::mma_ts(tmem + C::kTmemO, p_hi + BN / 2 + ks * 8, bdesc, idesc_pv, 1u);
            }
            tc::commit(&bars->p_free[pb]);
            // V (or, with k_eq_v, the whole K stage) is free once PV ends
            tc::commit(KEQV ? &bars->k_empty[vstage] : &bars->v_empty[g_tile % VS]);
            if (last) tc::commit(&bars->o_full);  // the item's O is final
          }
        }
      }
      if (!ok) {
        flag_error(err, PSW_DEVERR_PIPELINE);
        *abort_flag = 1;
      }
      // every MMA this thread issued has finished before tensor memory is freed
      tc::commit(&bars->mma_drained);
      mbar_wait(&bars->mma_drained, 0);
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    // Warp w owns the 32 rows of tensor-memory lane quadrant w and every key
    // column of a tile: a row's maximum and sum stay inside one thread.
    const int quad = warp;
    const int r = quad * 32 + lane;  // tile row
    const int t = r / group;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool use_cap = softcap > 0.f;
    const float sc = use_cap ? scale / softcap : 0.f;               // y = s_raw * sc
    const float mul = use_cap ? softcap * kLog2e : scale * kLog2e;  // log2-domain factor
    const uint64_t mul2 = f2_pack(mul, mul);
    // x-domain coefficients: x (A + x^2 (C1 + x^2 (C2 + x^2 C3))) = mul tanh(x sc)
    // to the y^7 term (with softcap), A x = mul x without
    const float A = use_cap ? sc * mul : mul;
    const float B = sc * sc;
    const float C1 = A * B * (-1.f / 3.f);
    const float C2 = A * B * B * (2.f / 15.f);
    const float C3 = A * B * B * B * (-17.f / 315.f);
    int g_tile = 0;  // global tile counter (S/P buffers, K/V stages)
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->item_full[slot], (n >> 1) & 1));
      const int item = ok ? bars->item[slot] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (!ok || item < 0) break;
      int kvh, dh;
      Geom g;
      item_geom(item, kvh, dh, g);
      const bool row_ok = t < g.tok_valid;
      const int p = g.past + g.i0 + t;
      const int vis_lo = (window > 0) ? max(0, p - window + 1) : 0;  // row sees [vis_lo, p]
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < g.nkt; ++j, ++g_tile) {
        const int sb = g_tile % C::kSP;
        // every decision below is warp-uniform
        ok = warp_wait(&bars->s_full[sb], (g_tile / C::kSP) & 1) && !*abort_flag;
        if (!ok) break;
        tc::fence_after();
        float x[BN];
        {
          uint32_t v[BN];
#pragma unroll
          for (int c16 = 0; c16 < BN / 16; ++c16)
            tc::ld16(tmem + lane_off + C::kTmemS + sb * BN + c16 * 16,
                     *reinterpret_cast<uint32_t(*)[16]>(&v[c16 * 16]));
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < BN; ++i) x[i] = __uint_as_float(v[i]);
        }

        const int key0 = (g.kt0 + j) * BN;
        const bool interior =
            __all_sync(0xffffffffu, row_ok && key0 >= vis_lo && key0 + BN - 1 <= p);
        // z: log2-domain exponent of P (score minus the running maximum).
        // Fast path (interior tile, every |s/cap| of the warp's tile <= 1/4):
        // the row maximum comes from the raw maximum (the softcap is monotone)
        // and z = x r(x^2) - m, the odd Taylor polynomial of tanh through y^7
        // (next term below 8.3e-8) with the scale, the softcap and log2 e
        // folded into its coefficients: five packed FMAs per pair.
        // Otherwise (edge tiles, larger |s/cap|) the capped scores are formed
        // first, hidden keys are set to -inf, and their maximum is taken.
        uint64_t z2[BN / 2];
        float alpha = 1.f;
        {
          const float mx = max_of<BN>(x);
          bool poly_ok = true;
          if (use_cap) {
            const float mn = min_of<BN>(x);
            // NaN (a never-cached slot beyond the sequence end, masked below)
            // must not force the slow path: compare with "not greater"
            poly_ok = __all_sync(0xffffffffu, !(fmaxf(mx, -mn) * sc > 0.25f));
          }
          const bool fast = interior && poly_ok;
          float tmax = 0.f;
          if (fast) tmax = use_cap ? mul * tanh_p7(mx * sc) : mx * mul;
          if (fast) {
            if (tmax > m_run + kRescaleThreshold) {  // lazy rescale (also the first key)
              // first visible keys of the row: O = 0, nothing to rescale
              alpha = (m_run == -INFINITY) ? 1.f : ex2_approx(m_run - tmax);
              m_run = (m_run == -INFINITY) ? tmax + kMaxBias : tmax;
            }
            log2_terms<BN>(x, z2, use_cap, A, C1, C2, C3, -m_run);
          } else {
            if (use_cap && poly_ok) {
              log2_terms<BN>(x, z2, true, A, C1, C2, C3, 0.f);
            } else if (use_cap) {
#pragma unroll
              for (int i = 0; i < BN / 2; ++i)
                z2[i] = f2_pack(mul * tanh_exp(x[2 * i] * sc), mul * tanh_exp(x[2 * i + 1] * sc));
            } else {
#pragma unroll
              for (int i = 0; i < BN / 2; ++i) z2[i] = f2_mul(f2_pack(x[2 * i], x[2 * i + 1]), mul2);
            }
            // columns [a, b] of the tile are visible to this row: one bit each
            uint64_t vis = 0;
            {
              const int a = vis_lo - key0, b = p - key0;
              if (row_ok && b >= 0 && a <= BN - 1) {
                const int a0 = a < 0 ? 0 : a, b0 = b > BN - 1 ? BN - 1 : b;
                vis = (~0ull >> (63 - b0)) & (~0ull << a0);
              }
            }
            float uu[BN];
#pragma unroll
            for (int i = 0; i < BN / 2; ++i) {
              const float2 w = f2_unpack(z2[i]);
              uu[2 * i] = (vis >> (2 * i)) & 1ull ? w.x : -INFINITY;
              uu[2 * i + 1] = (vis >> (2 * i + 1)) & 1ull ? w.y : -INFINITY;
            }
            tmax = max_of<BN>(uu);
            if (tmax > m_run + kRescaleThreshold) {
              alpha = (m_run == -INFINITY) ? 1.f : ex2_approx(m_run - tmax);
              m_run = (m_run == -INFINITY) ? tmax + kMaxBias : tmax;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            const uint64_t negm2 = f2_pack(-m_use, -m_use);
#pragma unroll
            for (int i = 0; i < BN / 2; ++i)
              z2[i] = f2_add(f2_pack(uu[2 * i], uu[2 * i + 1]), negm2);
          }
        }
        // rescaling O needs the item's previous PV finished
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const int gprev = g_tile - 1;
          ok = warp_wait(&bars->p_free[gprev % C::kSP], (gprev / C::kSP) & 1);
          if (!ok) break;
          tc::fence_after();
#pragma unroll 1
          for (int c16 = 0; c16 < C::kOCols / 16; ++c16) {
            const uint32_t col = tmem + lane_off + C::kTmemO + c16 * 16;
            uint32_t v[16];
            tc::ld16(col, v);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tc::st16(col, v);
          }
          tc::wait_st();
        }
        // with k_eq_v, V is this tile's K stage (landed: S was formed from it;
        // not reloaded before PV has read it): zero the rows of keys that no
        // row of the item may see on its first / last tile. A V tile of its
        // own is zeroed by the V producer before it is reported.
        if (KEQV && (j == 0 || j == g.nkt - 1)) {
          const int tkey0 = (g.kt0 + j) * BN;
          const int z_lo = max(0, g.j_lo - tkey0);       // rows [0, z_lo) hidden
          const int z_hi = min(BN, g.j_hi - tkey0 + 1);  // rows [z_hi, BN) hidden
          if (z_lo > 0 || z_hi < BN) {
            const int vstage = (g_tile * C::kKHalves + C::kKHalves - 1) % KS;
            uint8_t* vt = k_ring + vstage * C::kKBytes + (C::kSplitK ? 0 : dh * C::kVChunks * 1024);
            for (int idx = threadIdx.x; idx < C::kVChunks * BN * 8; idx += kSoftmaxWarps * 32) {
              const int cv = idx / (BN * 8);
              const int rem = idx - cv * (BN * 8);
              const int row = rem >> 3, uu = rem & 7;
              const int off = (row >> 3) * C::kKGroupBytes + cv * 1024 + (row & 7) * 128;
              if (row < z_lo || row >= z_hi)
                *reinterpret_cast<uint4*>(vt + off + uu * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
        }
        {
          // P = 2^z: bf16 high part and bf16 remainder into tensor memory, 16
          // column pairs at a time, each stage over 8 pairs before the next
          uint64_t ps2[2] = {0ull, 0ull};
          constexpr int kChunkPairs = (BN / 2 < 16) ? BN / 2 : 16;
          constexpr int G = 8;
#pragma unroll
          for (int c = 0; c < BN / 2 / kChunkPairs; ++c) {
            uint32_t hi[kChunkPairs], lo[kChunkPairs];
#pragma unroll
            for (int gb = 0; gb < kChunkPairs; gb += G) {
              float pa[G], pb[G];
#pragma unroll
              for (int k = 0; k < G; ++k) {
                const float2 z = f2_unpack(z2[c * kChunkPairs + gb + k]);
                pa[k] = ex2_approx(z.x);
                pb[k] = ex2_approx(z.y);
              }
#pragma unroll
              for (int k = 0; k < G; ++k) {
                const uint64_t ab = f2_pack(pa[k], pb[k]);
                ps2[k & 1] = f2_add(ps2[k & 1], ab);
                // P = hi + lo without conversion instructions: hi keeps the
                // upper 16 bits of P (bf16 by truncation), lo = P - hi exactly,
                // then truncated to bf16 the same way; together they carry P to
                // 2^-14 relative.
                hi[gb + k] = __byte_perm(__float_as_uint(pa[k]), __float_as_uint(pb[k]), 0x7632);
                const uint32_t ha = __float_as_uint(pa[k]) & 0xFFFF0000u;
                const uint32_t hb = __float_as_uint(pb[k]) & 0xFFFF0000u;
                const float2 l =
                    f2_unpack(f2_sub(ab, f2_pack(__uint_as_float(ha), __uint_as_float(hb))));
                lo[gb + k] = __byte_perm(__float_as_uint(l.x), __float_as_uint(l.y), 0x7632);
              }
            }
            const uint32_t pcol = tmem + lane_off + C::kTmemS + sb * BN + c * kChunkPairs;
            if constexpr (kChunkPairs == 16) {
              tc::st16(pcol, hi);
              tc::st16(pcol + BN / 2, lo);
            } else {
              tc::st8(pcol, *reinterpret_cast<uint32_t(*)[8]>(hi));
              tc::st8(pcol + BN / 2, *reinterpret_cast<uint32_t(*)[8]>(lo));
            }
          }
          const float2 ps_a = f2_unpack(ps2[0]), ps_b = f2_unpack(ps2[1]);
          l_run = l_run * alpha + ((ps_a.x + ps_a.y) + (ps_b.x + ps_b.y));
          tc::wait_st();
          tc::fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      // row maximum and sum for the epilogue warps (double-buffered by item)
      if (n >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->stats_free[slot], ((n >> 1) - 1) & 1));
        if (!ok) break;
      }
      bars->stat_m[slot][r] = m_run;
      bars->stat_l[slot][r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->stats_full[slot]);
    }
    if (!ok && lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp 4 + q writes the O rows of lane quadrant q once the item's last PV
    // is done, straight from tensor memory: each 16-lane half is read 32
    // columns at a time in the 16x256b shape, where four consecutive lanes
    // hold 8 consecutive columns of one row, so every store writes whole
    // 32-byte sectors; O is scaled by 1/l, lse = m + ln l. Meanwhile the
    // softmax warps already work on the next item.
    const int quad = warp - kSoftmaxWarps;  // = warp mod 4: its lane quadrant
    const int r = quad * 32 + lane;
    const int t = r / group;
    const int h = r - t * group;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->item_full[slot], (n >> 1) & 1));
      const int item = ok ? bars->item[slot] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[slot]);
      if (!ok || item < 0) break;
      int kvh, dh;
      Geom g;
      item_geom(item, kvh, dh, g);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_full, n & 1)) &&
           __all_sync(0xffffffffu, mbar_wait(&bars->stats_full[slot], (n >> 1) & 1)) &&
           !*abort_flag;
      if (!ok) break;
      // Is this the CTA's last item? Its K producer published the next item
      // (or the end mark) before it loaded this item's last tile.
      const int nslot = (n + 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->item_full[nslot], ((n + 1) >> 1) & 1));
      if (!ok) break;
      const bool last_item = bars->item[nslot] < 0;
      // this lane's own row (lse) and the four rows it stores (two per half)
      const float m_row = bars->stat_m[slot][r];
      const float l_row = bars->stat_l[slot][r];
      float inv[4];
      float* orow[4];
      bool valid[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tr = quad * 32 + (e >> 1) * 16 + (e & 1) * 8 + (lane >> 2);
        const float lr = bars->stat_l[slot][tr];
        inv[e] = (lr > 0.f) ? 1.f / lr : 0.f;
        const int tt = tr / group, hh = tr - tt * group;
        valid[e] = tt < g.tok_valid;
        orow[e] = out + (static_cast<int64_t>(g.q0 + g.i0 + tt) * n_q + kvh * group + hh) * HD +
                  dh * C::kOCols + 2 * (lane & 3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->stats_free[slot]);
      if (t < g.tok_valid && dh == 0 && lse != nullptr)
        lse[static_cast<int64_t>(g.q0 + g.i0 + t) * n_q + kvh * group + h] =
            (l_row > 0.f) ? (m_row + log2f(l_row)) * kLn2 : -INFINITY;
      tc::fence_after();
      if (last_item) {
        // Nothing follows this item: its last PV has completed, so every MMA
        // and TMA copy of the CTA has, and the Q/K/V rings are free. Each
        // thread stages its own row, scaled by 1/l, in shared memory (rows
        // 1040 B apart, so a warp's 16-byte stores fall in distinct banks)
        // and writes it with one bulk copy.
        constexpr int kRowStride = C::kOCols * 4 + 16;
        static_assert(kRows * kRowStride <= C::kQBytes + KS * C::kKBytes +
                                                 C::kVStages * C::kVBytes,
                      "staged output fits the rings");
        uint8_t* srow = smem + r * kRowStride;
        const float inv_r = (l_row > 0.f) ? 1.f / l_row : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < C::kOCols; c0 += 32) {
          uint32_t v[32];
          tc::ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kTmemO + c0, v);
          tc::wait_ld();
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float4 w;
            w.x = __uint_as_float(v[4 * q4]) * inv_r;
            w.y = __uint_as_float(v[4 * q4 + 1]) * inv_r;
            w.z = __uint_as_float(v[4 * q4 + 2]) * inv_r;
            w.w = __uint_as_float(v[4 * q4 + 3]) * inv_r;
            *reinterpret_cast<float4*>(srow + (c0 + 4 * q4) * 4) = w;
          }
        }
        if (t < g.tok_valid) {
          fence_proxy_async_smem();  // the bulk copy reads these rows
          bulk_store(out + (static_cast<int64_t>(g.q0 + g.i0 + t) * n_q + kvh * group + h) * HD +
                         dh * C::kOCols,
                     srow, C::kOCols * 4);
          bulk_commit();
          bulk_wait_read();
        }
      }
      // two 32-column blocks (four loads) in flight per wait
#pragma unroll 1
      for (int cb = 0; cb < C::kOCols / 32 && !last_item; cb += 2) {
        uint32_t v[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tc::ld16x256_x4(tmem + (static_cast<uint32_t>(quad * 32 + (q & 1) * 16) << 16) +
                              C::kTmemO + (cb + (q >> 1)) * 32,
                          v[q]);
        tc::wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int hf = q & 1, cc = cb + (q >> 1);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int e = hf * 2 + e2;
              if (valid[e]) {
                float2 w;
                w.x = __uint_as_float(v[q][4 * k + 2 * e2]) * inv[e];
                w.y = __uint_as_float(v[q][4 * k + 2 * e2 + 1]) * inv[e];
                *reinterpret_cast<float2*>(orow[e] + cc * 32 + 8 * k) = w;
              }
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free);
    }
    if (!ok && lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *abort_flag = 1;
    }
  }

done:
  tc::fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc::fence_after();
    tc::dealloc(tmem, C::kTmemCols);
  }
}

template <int HD, bool KEQV>
int launch(const LayerArgs& L, const CUtensorMap& q_map, const CUtensorMap& k_map,
           const CUtensorMap& v_map, const int32_t* cu_q, const int32_t* past_lens, int n_seqs,
           int n_q_total, int max_q_len, const int32_t* block_table, int max_blocks,
           int64_t num_blocks, float* out, float* lse, void* ws, int num_sms, int32_t* err,
           cudaStream_t stream) {
  using C = Cfg<HD, KEQV>;
  if (set_smem_limit(reinterpret_cast<const void*>(prefill_kernel<HD, KEQV>), C::kSmemBytes) !=
      PSW_OK)
    return PSW_ELAUNCH;
  const int T = kRows / L.group();
  const int max_rb = (max_q_len + T - 1) / T;
  // the work list sits after the counter block, which this call leaves alone
  uint8_t* wl = static_cast<uint8_t*>(ws) + kWsCounterBytes;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(wl);
  int2* units = reinterpret_cast<int2*>(wl + sizeof(PlanHeader));
  prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(cu_q, past_lens, n_seqs, n_q_total,
                                                      max_q_len, max_blocks, L.window, T, C::kBN,
                                                      max_rb, hdr, units, err);
  if (cudaGetLastError() != cudaSuccess) return PSW_ELAUNCH;
  const int64_t max_items =
      static_cast<int64_t>(n_seqs) * max_rb * L.n_kv * C::kDSplit;
  const int grid = static_cast<int>(max_items < num_sms ? max_items : num_sms);
  const StallHook stall = stall_hook(kStallPrefill);
  prefill_kernel<HD, KEQV><<<grid, kThreads, C::kSmemBytes, stream>>>(
      q_map, k_map, v_map, cu_q, past_lens, block_table, max_blocks, num_blocks, n_q_total,
      max_q_len, L.n_q, L.group(), L.window, L.scale, L.softcap, hdr, units, out, lse, err,
      stall.cta, stall.tile);
  return cudaGetLastError() == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace pf

size_t prefill_workspace_bytes(const LayerArgs& L, int n_seqs, int max_q_len) {
  const int T = pf::kRows / L.group();
  const size_t max_rb = (static_cast<size_t>(max_q_len > 0 ? max_q_len : 0) + T - 1) / T;
  const size_t bytes = kWsCounterBytes + sizeof(pf::PlanHeader) +
                       static_cast<size_t>(n_seqs) * max_rb * sizeof(int2);
  return (bytes + 255) / 256 * 256;
}

int launch_prefill(const LayerArgs& L, const CUtensorMap& q_map, const CUtensorMap& k_map,
                   const CUtensorMap& v_map, const int32_t* cu_q, const int32_t* past_lens,
                   int n_seqs, int n_q_total, int max_q_len, const int32_t* block_table,
                   int max_blocks, int64_t num_blocks, float* out, float* lse, void* ws,
                   int num_sms, int32_t* err, cudaStream_t stream) {
  if (L.hd == 256)
    return L.k_eq_v ? pf::launch<256, true>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                            n_q_total, max_q_len, block_table, max_blocks,
                                            num_blocks, out, lse, ws, num_sms, err, stream)
                    : pf::launch<256, false>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                             n_q_total, max_q_len, block_table, max_blocks,
                                             num_blocks, out, lse, ws, num_sms, err, stream);
  return L.k_eq_v ? pf::launch<512, true>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                          n_q_total, max_q_len, block_table, max_blocks,
                                          num_blocks, out, lse, ws, num_sms, err, stream)
                  : pf::launch<512, false>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                           n_q_total, max_q_len, block_table, max_blocks,
                                           num_blocks, out, lse, ws, num_sms, err, stream);
}

}  // namespace psw
