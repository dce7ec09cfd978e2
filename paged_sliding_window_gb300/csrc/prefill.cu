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
// Design (how, on sm_103a), one CTA per (sequence, KV head, block of 128/G
// chunk tokens, half of head_dim for head_dim 512):
//  * 128 query rows = (128/G tokens) x (G heads), token-major. Q is loaded once
//    by TMA (128-byte swizzle, one box per 64 columns of head_dim).
//  * Warps 8 (Q, K) and 10 (V) stream K and V tiles of BN keys (64 for
//    head_dim 256, 32 for 512) into rings of their own (3 K and 2 V stages
//    where shared memory allows), one 2 KB TMA box per (page, 64-column
//    chunk), and warm L2 with the tile three ahead. A K stage is released as
//    soon as QK has read it, a V stage after PV. Pages past the sequence end
//    load as zeros.
//  * Warp 9 (one elected thread) issues tcgen05.mma: S_j = Q K_j^T (SS, both
//    K-major) into one of two S buffers in TMEM, and O += P_j V_j (TS: P from
//    one of two P buffers in TMEM, V MN-major from shared memory). The issue
//    order QK_0, QK_1, PV_0, QK_2, PV_1, ... keeps the tensor pipe fed while
//    the softmax warps work on the tile before.
//  * Warps 0-7 run the softmax. Warps w and w+4 own the same 32 rows (TMEM
//    lanes 32 (w mod 4) ...) and split the BN key columns in halves; per tile
//    they exchange one partial row maximum through shared memory. Scores get
//    scale, softcap (odd polynomial on the FMA pipe for |s/cap| <= 1/2, the
//    exp formula beyond) and, on band-edge tiles only, the band/causal
//    predicate; the online softmax runs in fp32 in the exp2 domain with lazy
//    rescaling of O (only when the running max grows by more than 2^8; the
//    two warps of a row pair rescale half of O each). P is written back to
//    TMEM as a bf16 high part and a bf16 remainder, split with integer ops
//    (no conversion instructions); both are multiplied into O, so P enters the
//    product to 2^-14 relative.
//  * V rows of key positions that no row of the tile can see (before the
//    window of the tile's first row, after its last row) are zeroed in shared
//    memory so uncached or stale slots never reach O.
//  * Every wait is bounded; on timeout the kernel flags PSW_DEVERR_PIPELINE,
//    drains its own copies and MMAs, frees its tensor memory and returns.
#include <math.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace pf {

constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;   // Q and K tiles
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10; // V tiles (idle with k_eq_v)
constexpr int kThreads = 11 * 32;
constexpr int kRows = 128;
constexpr int kPageBoxBytes = kBlockSize * 128;  // one TMA box: 16 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int HD, bool KEQV>
struct Cfg {
  static constexpr int kQChunks = HD / 64;
  static constexpr int kBN = (HD == 256) ? 64 : 32;
  static constexpr int kHalf = kBN / 2;  // key columns per softmax warp
  static constexpr int kPagesPerTile = kBN / kBlockSize;
  static constexpr int kOCols = 256;
  static constexpr int kDSplit = HD / kOCols;
  static constexpr int kVChunks = kOCols / 64;
  static constexpr int kQBytes = kQChunks * kRows * 128;
  static constexpr int kChunkTileBytes = kBN * 128;  // one 64-column chunk of a K/V tile
  static constexpr int kKBytes = kQChunks * kChunkTileBytes;
  static constexpr int kVBytes = KEQV ? 0 : kVChunks * kChunkTileBytes;
  static constexpr int kBarsBytes = 1536;
  static constexpr int kBudget = 232448 - 1024 - kQBytes - kBarsBytes;
  // K and V have rings of their own: K is consumed early (QK), V late (PV).
  // Three K stages where they fit (two for head_dim 512 without k_eq_v), two
  // V stages (one when only that fits).
  static constexpr int kKStages = (3 * kKBytes + 2 * kVBytes <= kBudget) ? 3 : 2;
  static constexpr int kVStages = KEQV ? 0 : ((kKStages * kKBytes + 2 * kVBytes <= kBudget) ? 2 : 1);
  static constexpr int kSmemBytes =
      1024 + kQBytes + kKStages * kKBytes + kVStages * kVBytes + kBarsBytes;
  static constexpr int kVS = kVStages > 0 ? kVStages : 1;  // ring size for index math
  // tensor memory columns: O | S0 | S1 | P0 (hi, lo) | P1 (hi, lo)
  static constexpr int kTmemO = 0;
  static constexpr int kTmemS = 256;                 // + b * kBN
  static constexpr int kTmemP = 256 + 2 * kBN;       // + b * kBN; hi then lo (kBN/2 each)
  static constexpr int kTmemCols = 512;
  static constexpr int kTmaPerStage = kPagesPerTile * (kQChunks + (KEQV ? 0 : kVChunks));
  static_assert(kTmaPerStage <= 32, "one TMA box per producer lane");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kTmemP + 2 * kBN <= kTmemCols, "tensor memory columns");
  static_assert(kKStages * kKBytes + kVStages * kVBytes <= kBudget, "K/V rings");
};

template <int S>
__device__ __forceinline__ int stage_of(int j) { return j % S; }
template <int S>
__device__ __forceinline__ uint32_t round_of(int j) { return static_cast<uint32_t>(j / S) & 1u; }

struct Bars {
  uint64_t q_full;
  // K and V rings are filled and released separately: a K stage is free once
  // QK has read it, a V stage once PV has (with k_eq_v, V is the K stage and
  // it is released after PV). First kKStages / kVStages entries used.
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t mma_drained;
  uint32_t tmem_base;
  int abort;     // set by any warp; read by the producer and the MMA issuer
  int sm_abort;  // set only by softmax threads, read after their named barrier
  float red[2][kRows];  // [column half][row]: partial row max per tile, then row sums
};

// tanh(y) for |y| <= 1/2: odd Taylor polynomial through y^11 (the next term
// is below 4.4e-7). Branch-free, FMA pipe only.
__device__ __forceinline__ float tanh_small(float y) {
  const float y2 = y * y;
  float r = -1382.f / 155925.f;
  r = fmaf(r, y2, 62.f / 2835.f);
  r = fmaf(r, y2, -17.f / 315.f);
  r = fmaf(r, y2, 2.f / 15.f);
  r = fmaf(r, y2, -1.f / 3.f);
  return fmaf(r * y2, y, y);
}

// tanh_small on a pair of values (packed fp32 arithmetic).
__device__ __forceinline__ uint64_t tanh_small2(uint64_t y) {
  const uint64_t y2 = f2_mul(y, y);
  uint64_t r = f2_fma(f2_pack(-1382.f / 155925.f, -1382.f / 155925.f), y2,
                      f2_pack(62.f / 2835.f, 62.f / 2835.f));
  r = f2_fma(r, y2, f2_pack(-17.f / 315.f, -17.f / 315.f));
  r = f2_fma(r, y2, f2_pack(2.f / 15.f, 2.f / 15.f));
  r = f2_fma(r, y2, f2_pack(-1.f / 3.f, -1.f / 3.f));
  return f2_fma(f2_mul(r, y2), y, y);
}

// tanh(y) for any y: 1 - 2 / (e^{2|y|} + 1) with the sign restored, the
// polynomial where |y| <= 1/2 (where this form loses relative precision).
__device__ __forceinline__ float tanh_any(float y) {
  const float ay = fabsf(y);
  const float t = ex2_approx(-2.f * kLog2e * ay);  // e^{-2|y|}
  const float big = copysignf(__fdividef(1.f - t, 1.f + t), y);
  return ay <= 0.5f ? tanh_small(y) : big;
}

template <int HD, bool KEQV>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
               const __grid_constant__ CUtensorMap v_map, const int32_t* __restrict__ cu_q,
               const int32_t* __restrict__ past_lens, const int32_t* __restrict__ block_table,
               int max_blocks, int64_t num_blocks, int n_q_total, int max_q_len, int n_q,
               int group, int window, float scale, float softcap, float* __restrict__ out,
               float* __restrict__ lse, int32_t* err) {
  using C = Cfg<HD, KEQV>;
  constexpr int BN = C::kBN;
  constexpr int HALF = C::kHalf;
  const int T = kRows / group;  // chunk tokens per tile
  const int rb = blockIdx.x;
  const int kvh = blockIdx.y / C::kDSplit;
  const int dh = blockIdx.y - kvh * C::kDSplit;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- tile geometry (uniform across the CTA)
  const int q0 = cu_q[b];
  int n_b = cu_q[b + 1] - q0;
  const int past = past_lens[b];
  if (n_b < 0 || past < 0 || q0 < 0) {
    if (rb == 0 && threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PSW_DEVERR_LENGTH);
    return;
  }
  if (n_b > max_q_len || q0 + n_b > n_q_total) {
    if (rb == 0 && threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PSW_DEVERR_LENGTH);
    n_b = min(max_q_len, n_q_total - q0);
  }
  const int i0 = rb * T;
  if (i0 >= n_b) return;
  const int tok_valid = min(T, n_b - i0);
  const int p_lo = past + i0;
  const int p_hi = past + i0 + tok_valid - 1;
  const int seq_end = past + n_b;  // positions < seq_end are cached
  if (static_cast<int64_t>(seq_end) > static_cast<int64_t>(max_blocks) * kBlockSize) {
    if (rb == 0 && threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PSW_DEVERR_CAPACITY);
  }
  const int j_lo = (window > 0) ? max(0, p_lo - window + 1) : 0;
  const int j_hi = p_hi;
  const int kt0 = j_lo / BN;
  const int nkt = j_hi / BN - kt0 + 1;
  const int last_page = min((seq_end - 1) / kBlockSize, max_blocks - 1);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem;
  uint8_t* k_ring = smem + C::kQBytes;
  uint8_t* v_ring = k_ring + C::kKStages * C::kKBytes;
  Bars* bars = reinterpret_cast<Bars*>(v_ring + C::kVStages * C::kVBytes);
  static_assert(sizeof(Bars) <= C::kBarsBytes, "barrier block");

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], kSoftmaxWarps);
      mbar_init(&bars->p_full[i], kSoftmaxWarps);
      mbar_init(&bars->p_free[i], 1);
    }
    mbar_init(&bars->mma_drained, 1);
    bars->abort = 0;
    bars->sm_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(&bars->tmem_base, C::kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ------------------------------------------------------------ producers
    const bool v_side = (warp == kVProducerWarp);
    if (v_side && KEQV) goto done;  // V is the K tile
    if (!v_side && lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      if (!KEQV) prefetch_tensormap(&v_map);
      mbar_arrive_expect_tx(&bars->q_full,
                            static_cast<uint32_t>(C::kQChunks * group * T * 128));
      for (int c = 0; c < C::kQChunks; ++c)
        tma_load_3d(q_smem + c * (kRows * 128), &q_map, &bars->q_full, c * 64, kvh * group,
                    q0 + i0);
    }
    // K boxes: lane -> (page, chunk) for lane < pages * kQChunks; V boxes likewise
    const int k_lp = lane / C::kQChunks, k_lc = lane - k_lp * C::kQChunks;
    const int v_lp = lane / C::kVChunks, v_lc = lane - v_lp * C::kVChunks;
    constexpr int kKBoxes = C::kPagesPerTile * C::kQChunks;
    constexpr int kVBoxes = C::kPagesPerTile * C::kVChunks;
    // Block ids of this CTA's pages, 32 at a time: lane l holds page
    // first_page + 32 g + l of group g; the next group is loaded one group
    // ahead, so a tile needs only shuffles.
    constexpr int P = C::kPagesPerTile;
    constexpr int kTilesPerGroup = 32 / P;
    const int first_page = kt0 * P;
    auto load_group = [&](int grp) -> int {
      const int page = first_page + grp * 32 + lane;
      if (grp * kTilesPerGroup >= nkt || page > last_page) return -1;
      int blk = block_table[static_cast<int64_t>(b) * max_blocks + page];
      if (blk < 0 || blk >= num_blocks) {
        flag_error(err, PSW_DEVERR_BLOCK_ID);
        blk = -1;  // out-of-range box: TMA fills zeros
      }
      return blk;
    };
    int ids = load_group(0), ids_next = load_group(1);
    const int nst = v_side ? C::kVS : C::kKStages;
    const int my_lp = v_side ? v_lp : k_lp;
    int issued = 0;
    for (int j = 0; j < nkt; ++j, ++issued) {
      const int stage = j % nst;
      const uint32_t ph = static_cast<uint32_t>(j / nst) & 1u;
      if (j > 0 && j % kTilesPerGroup == 0) {
        ids = ids_next;
        ids_next = load_group(j / kTilesPerGroup + 1);
      }
      const int src = (j % kTilesPerGroup) * P + (my_lp < P ? my_lp : 0);
      const int my_blk = __shfl_sync(0xffffffffu, ids, src);
      const int jp = j + 3;  // tile whose pages are warmed in L2 now
      const int psrc = (jp % kTilesPerGroup) * P + (my_lp < P ? my_lp : 0);
      const int pf_same = __shfl_sync(0xffffffffu, ids, psrc);
      const int pf_next = __shfl_sync(0xffffffffu, ids_next, psrc);
      const int pf_blk = (jp / kTilesPerGroup == j / kTilesPerGroup) ? pf_same : pf_next;
      uint64_t* empty = v_side ? &bars->v_empty[stage] : &bars->k_empty[stage];
      uint64_t* full = v_side ? &bars->v_full[stage] : &bars->k_full[stage];
      bool ok = true;
      if (lane == 0) ok = mbar_wait(empty, ph ^ 1);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag) {
        if (lane == 0) { flag_error(err, PSW_DEVERR_PIPELINE); *abort_flag = 1; }
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(full, v_side ? C::kVBytes : C::kKBytes);
      __syncwarp();
      if (!v_side) {
        if (lane < kKBoxes) {
          tma_load_3d(k_ring + stage * C::kKBytes + k_lc * C::kChunkTileBytes +
                          k_lp * kPageBoxBytes,
                      &k_map, full, 0, kvh * C::kQChunks + k_lc, my_blk * kBlockSize);
          if (jp < nkt && pf_blk >= 0)  // warm L2 with the tile three ahead
            tma_prefetch_3d(&k_map, 0, kvh * C::kQChunks + k_lc, pf_blk * kBlockSize);
        }
      } else {
        if (lane < kVBoxes) {
          const int y = kvh * C::kQChunks + dh * C::kVChunks + v_lc;
          tma_load_3d(v_ring + stage * C::kVBytes + v_lc * C::kChunkTileBytes +
                          v_lp * kPageBoxBytes,
                      &v_map, full, 0, y, my_blk * kBlockSize);
          if (jp < nkt && pf_blk >= 0) tma_prefetch_3d(&v_map, 0, y, pf_blk * kBlockSize);
        }
      }
    }
    if (lane == 0) {  // drain this warp's own copies before anyone leaves
      if (!v_side) mbar_wait(&bars->q_full, 0);
      for (int i = max(0, issued - nst); i < issued; ++i)
        mbar_wait(v_side ? &bars->v_full[i % nst] : &bars->k_full[i % nst],
                  static_cast<uint32_t>(i / nst) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, BN, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, C::kOCols, 0, 1);
      const uint32_t q_base = smem_u32(q_smem);
      const uint32_t k_base = smem_u32(k_ring);
      const uint32_t v_base = smem_u32(v_ring);
      bool ok = mbar_wait(&bars->q_full, 0);
      // Non-blocking scheduler: issue QK_j as soon as K_j has landed and its S
      // buffer is free (at most two ahead of the softmax), PV_i as soon as P_i
      // is in TMEM and V_i has landed; QK first, so S is ready before the
      // softmax asks for it. The tensor pipe runs the MMAs in issue order.
      int next_qk = 0, next_pv = 0;
      long long idle_since = clock64();
      while (ok && next_pv < nkt) {
        bool progressed = false;
        if (next_qk < nkt && next_qk < next_pv + 2) {
          const int j = next_qk, sb = j & 1;
          if (mbar_try_wait(&bars->k_full[stage_of<C::kKStages>(j)], round_of<C::kKStages>(j)) &&
              (j < 2 || mbar_try_wait(&bars->s_free[sb], ((j >> 1) - 1) & 1))) {
            tc::fence_after();
            const uint32_t kb = k_base + stage_of<C::kKStages>(j) * C::kKBytes;
            #pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              const int c = ks >> 2;
              const uint64_t adesc = tc::smem_desc(q_base + c * (kRows * 128) + (ks & 3) * 32,
                                                   16, 1024, tc::kSwizzle128B);
              const uint64_t bdesc = tc::smem_desc(kb + c * C::kChunkTileBytes + (ks & 3) * 32,
                                                   16, 1024, tc::kSwizzle128B);
              tc::mma_ss(tmem + C::kTmemS + sb * BN, adesc, bdesc, idesc_qk, ks > 0 ? 1u : 0u);
            }
            tc::commit(&bars->s_full[sb]);
            if (!KEQV) tc::commit(&bars->k_empty[stage_of<C::kKStages>(j)]);  // K read by QK
            ++next_qk;
            progressed = true;
          }
        }
        if (!progressed && next_pv < next_qk) {
          const int i = next_pv, pb = i & 1;
          if (mbar_try_wait(&bars->p_full[pb], (i >> 1) & 1) &&
              (KEQV || mbar_try_wait(&bars->v_full[stage_of<C::kVS>(i)], round_of<C::kVS>(i)))) {
            tc::fence_after();
            const uint32_t vb =
                KEQV ? k_base + stage_of<C::kKStages>(i) * C::kKBytes +
                           dh * C::kVChunks * C::kChunkTileBytes
                     : v_base + stage_of<C::kVS>(i) * C::kVBytes;
            const uint32_t p_hi = tmem + C::kTmemP + pb * BN;
            #pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
              const uint64_t bdesc = tc::smem_desc(vb + ks * 16 * 128, C::kChunkTileBytes, 1024,
                                                   tc::kSwizzle128B);
              tc::mma_ts(tmem + C::kTmemO, p_hi + ks * 8, bdesc, idesc_pv,
                         (i > 0 || ks > 0) ? 1u : 0u);
              tc::mma_ts(tmem + C::kTmemO, p_hi + BN / 2 + ks * 8, bdesc, idesc_pv, 1u);
            }
            tc::commit(&bars->p_free[pb]);
            // V (or, with k_eq_v, the whole K part) of this stage is free once PV ends
            tc::commit(KEQV ? &bars->k_empty[stage_of<C::kKStages>(i)]
                            : &bars->v_empty[stage_of<C::kVS>(i)]);
            ++next_pv;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = clock64();
        } else if (*abort_flag || clock64() - idle_since > kWaitLimitCycles) {
          ok = false;
        }
      }
      if (!ok) { flag_error(err, PSW_DEVERR_PIPELINE); *abort_flag = 1; }
      // every MMA this thread issued has finished before tensor memory is freed
      tc::commit(&bars->mma_drained);
      mbar_wait(&bars->mma_drained, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;       // TMEM lane quadrant = rows 32*quad ...
    const int half = warp >> 2;      // key columns [half*HALF, (half+1)*HALF)
    const int r = quad * 32 + lane;  // tile row
    const int t = r / group;
    const int h = r - t * group;
    const bool row_ok = (t < tok_valid) && (r < group * T);
    const int p = past + i0 + t;
    const int vis_lo = (window > 0) ? max(0, p - window + 1) : 0;  // this row sees [vis_lo, p]
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool use_cap = softcap > 0.f;
    const float inv_cap = use_cap ? 1.f / softcap : 0.f;
    const float scale_l2 = scale * kLog2e;
    const float mul = use_cap ? softcap * kLog2e : 1.f;  // log2-domain value of the proxy
    float m_run = -INFINITY, l_run = 0.f;
    volatile int* sm_abort = &bars->sm_abort;
    const uint32_t pair_bar = 1 + quad;  // named barrier of warps quad and quad + 4
    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      // every decision below is warp-uniform; the abort decision is taken by all
      // softmax warps together after the named barrier at the end of the tile
      bool okw = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sb], (j >> 1) & 1));
      const int key0 = (kt0 + j) * BN + half * HALF;
      float x[HALF];
      float alpha = 1.f;
      if (okw) {
        tc::fence_after();
        {
          uint32_t v[HALF];
          #pragma unroll
          for (int c16 = 0; c16 < HALF / 16; ++c16)
            tc::ld16(tmem + lane_off + C::kTmemS + sb * BN + half * HALF + c16 * 16,
                     *reinterpret_cast<uint32_t(*)[16]>(&v[c16 * 16]));
          tc::wait_ld();
          #pragma unroll
          for (int i = 0; i < HALF; ++i) x[i] = __uint_as_float(v[i]);
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[sb]);

        // scores to a monotone proxy u with log2-domain value mul * u: the tanh
        // of the softcap (mul = cap log2 e) or the scaled score (mul = 1);
        // every loop is branch-free
        if (use_cap) {
          const float sc = scale * inv_cap;
          const uint64_t sc2 = f2_pack(sc, sc);
          float amax = 0.f;
          #pragma unroll
          for (int i = 0; i < HALF / 2; ++i) {
            const float2 y = f2_unpack(f2_mul(f2_pack(x[2 * i], x[2 * i + 1]), sc2));
            x[2 * i] = y.x;
            x[2 * i + 1] = y.y;
            amax = fmaxf(amax, fmaxf(fabsf(y.x), fabsf(y.y)));
          }
          if (__any_sync(0xffffffffu, amax > 0.5f)) {
            #pragma unroll
            for (int k = 0; k < HALF; ++k) x[k] = tanh_any(x[k]);
          } else {
            #pragma unroll
            for (int i = 0; i < HALF / 2; ++i) {
              const float2 t = f2_unpack(tanh_small2(f2_pack(x[2 * i], x[2 * i + 1])));
              x[2 * i] = t.x;
              x[2 * i + 1] = t.y;
            }
          }
        } else {
          const uint64_t s2 = f2_pack(scale_l2, scale_l2);
          #pragma unroll
          for (int i = 0; i < HALF / 2; ++i) {
            const float2 t = f2_unpack(f2_mul(f2_pack(x[2 * i], x[2 * i + 1]), s2));
            x[2 * i] = t.x;
            x[2 * i + 1] = t.y;
          }
        }
        // band + causal predicate only where the tile straddles this row's edges
        const bool interior = row_ok && key0 >= vis_lo && key0 + HALF - 1 <= p;
        if (!__all_sync(0xffffffffu, interior)) {
          #pragma unroll
          for (int k = 0; k < HALF; ++k) {
            const int key = key0 + k;
            x[k] = (row_ok && key >= vis_lo && key <= p) ? x[k] : -INFINITY;
          }
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        #pragma unroll
        for (int k = 0; k < HALF; ++k) m4[k & 3] = fmaxf(m4[k & 3], x[k]);
        bars->red[half][r] = mul * fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      named_bar_sync(pair_bar, 64);  // the two halves of these rows meet
      if (okw) {
        const float m_tile = fmaxf(bars->red[0][r], bars->red[1][r]);
        if (m_tile > m_run + kRescaleThreshold) {  // lazy rescale (also the first visible key)
          alpha = ex2_approx(m_run - m_tile);
          m_run = m_tile;
        }
        // rescaling O needs PV_{j-1} finished; each warp of the pair takes half of O
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          okw = __all_sync(0xffffffffu,
                           mbar_wait(&bars->p_free[(j - 1) & 1], ((j - 1) >> 1) & 1));
          tc::fence_after();
          if (okw) {
            #pragma unroll 1
            for (int c16 = 0; c16 < C::kOCols / 32; ++c16) {
              const uint32_t col = tmem + lane_off + C::kTmemO + half * (C::kOCols / 2) + c16 * 16;
              uint32_t v[16];
              tc::ld16(col, v);
              tc::wait_ld();
              #pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tc::st16(col, v);
            }
            tc::wait_st();
          }
        }
      }
      if (okw) {
        // zero V rows that no row of this tile can see (first / last key tile)
        if (j == 0 || j == nkt - 1) {
          const int tkey0 = (kt0 + j) * BN;
          uint8_t* vt = KEQV ? k_ring + stage_of<C::kKStages>(j) * C::kKBytes +
                                   dh * C::kVChunks * C::kChunkTileBytes
                             : v_ring + stage_of<C::kVS>(j) * C::kVBytes;
          const int z_lo = max(0, j_lo - tkey0);       // rows [0, z_lo) hidden
          const int z_hi = min(BN, j_hi - tkey0 + 1);  // rows [z_hi, BN) hidden
          if (!KEQV && (z_lo > 0 || z_hi < BN))  // V may land after K
            okw = __all_sync(0xffffffffu, mbar_wait(&bars->v_full[stage_of<C::kVS>(j)],
                                                    round_of<C::kVS>(j)));
          if (okw && (z_lo > 0 || z_hi < BN)) {
            for (int idx = threadIdx.x; idx < C::kVChunks * BN * 8; idx += kSoftmaxWarps * 32) {
              const int cv = idx / (BN * 8);
              const int rem = idx - cv * (BN * 8);
              const int row = rem >> 3, u = rem & 7;
              if (row < z_lo || row >= z_hi)
                *reinterpret_cast<uint4*>(vt + cv * C::kChunkTileBytes + row * 128 + u * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
        }
        // P_{j-2} must have been multiplied in before its buffer is rewritten
        if (j >= 2)
          okw = __all_sync(0xffffffffu,
                           mbar_wait(&bars->p_free[sb], ((j >> 1) - 1) & 1));
      }
      if (okw) {
        // P = 2^(x - m): bf16 high part and bf16 remainder into tensor memory
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t mul2 = f2_pack(mul, mul), negm2 = f2_pack(-m_use, -m_use);
        uint64_t ps2[2] = {0ull, 0ull};
        uint32_t hi[HALF / 2], lo[HALF / 2];
        #pragma unroll
        for (int i = 0; i < HALF / 2; ++i) {
          const float2 z = f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), mul2, negm2));
          const float a = ex2_approx(z.x), bb = ex2_approx(z.y);
          const uint64_t ab = f2_pack(a, bb);
          ps2[i & 1] = f2_add(ps2[i & 1], ab);
          // P = hi + lo without conversion instructions: hi keeps the upper 16
          // bits of P (bf16 by truncation), lo = P - hi exactly, then truncated
          // to bf16 the same way; together they carry P to 2^-14 relative.
          const uint32_t ha = __float_as_uint(a) & 0xFFFF0000u;
          const uint32_t hb = __float_as_uint(bb) & 0xFFFF0000u;
          hi[i] = __byte_perm(ha, hb, 0x7632);
          const float2 l = f2_unpack(f2_sub(ab, f2_pack(__uint_as_float(ha), __uint_as_float(hb))));
          lo[i] = __byte_perm(__float_as_uint(l.x), __float_as_uint(l.y), 0x7632);
        }
        const float2 ps_a = f2_unpack(ps2[0]), ps_b = f2_unpack(ps2[1]);
        float ps[4] = {ps_a.x, ps_a.y, ps_b.x, ps_b.y};
        const uint32_t pcol = tmem + lane_off + C::kTmemP + sb * BN + half * (HALF / 2);
        if constexpr (HALF / 2 == 16) {
          tc::st16(pcol, hi);
          tc::st16(pcol + BN / 2, lo);
        } else {
          tc::st8(pcol, hi);
          tc::st8(pcol + BN / 2, lo);
        }
        l_run = l_run * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        tc::wait_st();
        tc::fence_before();
      }
      if (!okw && lane == 0) {
        flag_error(err, PSW_DEVERR_PIPELINE);
        *sm_abort = 1;
      }
      named_bar_sync(9, kSoftmaxWarps * 32);  // all softmax warps: V zeroing done, abort agreed
      if (*sm_abort) break;
      if (lane == 0) mbar_arrive(&bars->p_full[sb]);
    }
    bool ok = !*sm_abort;

    // epilogue: l from both halves, O / l staged through shared memory (the Q
    // tile and the K/V rings are idle once the last PV is done) and written out
    // as whole rows with coalesced stores, lse
    bars->red[half][r] = l_run;
    if (ok) ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars->p_free[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1));
    named_bar_sync(pair_bar, 64);
    tc::fence_after();
    const float l_tot = bars->red[0][r] + bars->red[1][r];
    const float inv_l = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
    // staging rows of kOCols floats plus 16 bytes of padding: 32 lanes storing
    // 16 bytes each at the same column of 32 rows then take the minimum four
    // shared-memory wavefronts
    constexpr int kORow = C::kOCols * 4 + 16;
    static_assert(kRows * kORow <= C::kQBytes + C::kKStages * C::kKBytes +
                                       C::kVStages * C::kVBytes,
                  "O staging fits in the Q tile and the K/V rings");
    uint8_t* ostage = q_smem;  // Q, then the K and V rings: contiguous and idle now
    if (ok) {
      #pragma unroll 1
      for (int c16 = 0; c16 < C::kOCols / 32; ++c16) {
        const int col0 = half * (C::kOCols / 2) + c16 * 16;
        uint32_t v[16];
        tc::ld16(tmem + lane_off + C::kTmemO + col0, v);
        tc::wait_ld();
        #pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float4 w;
          w.x = __uint_as_float(v[4 * q4 + 0]) * inv_l;
          w.y = __uint_as_float(v[4 * q4 + 1]) * inv_l;
          w.z = __uint_as_float(v[4 * q4 + 2]) * inv_l;
          w.w = __uint_as_float(v[4 * q4 + 3]) * inv_l;
          *reinterpret_cast<float4*>(ostage + r * kORow + (col0 + 4 * q4) * 4) = w;
        }
      }
      if (row_ok && dh == 0 && half == 0 && lse != nullptr)
        lse[static_cast<int64_t>(q0 + i0 + t) * n_q + kvh * group + h] =
            (l_tot > 0.f) ? (m_run + log2f(l_tot)) * kLn2 : -INFINITY;
    } else if (lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *abort_flag = 1;  // stops the producer and the MMA issuer
    }
    named_bar_sync(9, kSoftmaxWarps * 32);  // the whole O tile is staged
    if (ok) {
      // warp w copies rows w, w + 8, ...: 32 lanes x 16 bytes per store
      const int rows_valid = min(group * T, tok_valid * group);
      for (int rr = warp; rr < rows_valid; rr += kSoftmaxWarps) {
        const int tt = rr / group, hh = rr - tt * group;
        float* orow = out + (static_cast<int64_t>(q0 + i0 + tt) * n_q + kvh * group + hh) * HD +
                      dh * C::kOCols;
        #pragma unroll
        for (int c = lane; c < C::kOCols / 4; c += 32)
          reinterpret_cast<float4*>(orow)[c] =
              *reinterpret_cast<const float4*>(ostage + rr * kORow + c * 16);
      }
    }
  }

done:
  tc::fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, C::kTmemCols);
  }
}

template <int HD, bool KEQV>
int launch(const LayerArgs& L, const CUtensorMap& q_map, const CUtensorMap& k_map,
           const CUtensorMap& v_map, const int32_t* cu_q, const int32_t* past_lens, int n_seqs,
           int n_q_total, int max_q_len, const int32_t* block_table, int max_blocks,
           int64_t num_blocks, float* out, float* lse, int32_t* err, cudaStream_t stream) {
  using C = Cfg<HD, KEQV>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_kernel<HD, KEQV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return PSW_ELAUNCH;
    attr_set[dev] = true;
  }
  const int T = kRows / L.group();
  dim3 grid((max_q_len + T - 1) / T, L.n_kv * C::kDSplit, n_seqs);
  prefill_kernel<HD, KEQV><<<grid, kThreads, C::kSmemBytes, stream>>>(
      q_map, k_map, v_map, cu_q, past_lens, block_table, max_blocks, num_blocks, n_q_total,
      max_q_len, L.n_q, L.group(), L.window, L.scale, L.softcap, out, lse, err);
  return cudaGetLastError() == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace pf

int launch_prefill(const LayerArgs& L, const CUtensorMap& q_map, const CUtensorMap& k_map,
                   const CUtensorMap& v_map, const int32_t* cu_q, const int32_t* past_lens,
                   int n_seqs, int n_q_total, int max_q_len, const int32_t* block_table,
                   int max_blocks, int64_t num_blocks, float* out, float* lse, int32_t* err,
                   cudaStream_t stream) {
  if (L.hd == 256)
    return L.k_eq_v ? pf::launch<256, true>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                            n_q_total, max_q_len, block_table, max_blocks,
                                            num_blocks, out, lse, err, stream)
                    : pf::launch<256, false>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                             n_q_total, max_q_len, block_table, max_blocks,
                                             num_blocks, out, lse, err, stream);
  return L.k_eq_v ? pf::launch<512, true>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                          n_q_total, max_q_len, block_table, max_blocks,
                                          num_blocks, out, lse, err, stream)
                  : pf::launch<512, false>(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs,
                                           n_q_total, max_q_len, block_table, max_blocks,
                                           num_blocks, out, lse, err, stream);
}

}  // namespace psw
