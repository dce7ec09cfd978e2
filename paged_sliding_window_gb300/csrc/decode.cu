// decode.cu -- split-KV flash decoding over 16-token pages.
//
// Method (what is computed): for each sequence b and query head h, the single
// query at position p = seq_len - 1 attends over keys j <= p that the sliding
// window leaves visible (p - j < W, i.e. only the last min(seq_len, W) keys:
// InfiniLM PR 581 "feat: support gemma2 and gemma3_text", Gemma-3 item 3),
// with s = scale * q.k, the optional softcap cap * tanh(s / cap) on the scaled
// score before the softmax (same PR, Gemma-2 item 1), and V read from the K
// pages when k_eq_v ("MNN supports the full Gemma4 family", section 6.2).
// Keys are fetched through the block table of "Gemma 4 model architecture
// analysis" (vLLM-Kunlun), sections 6.3 and 6.5.
//
// Design (how, on sm_103a):
//  * Work unit = (sequence, KV head, group of <= 8 query heads); a unit's
//    visible pages are cut into tiles of 32 KB of K/V (2 pages at head_dim
//    256). All tiles of all units form one list, planned on the device from
//    seq_lens, and a persistent grid (two CTAs per SM) takes equal contiguous
//    slices of it, so the load is balanced whatever the length mix.
//  * Warp 4 is the producer: it reads block ids and issues one 2 KB TMA box
//    per (page, 128-byte chunk of head_dim) into a 3-stage shared-memory ring
//    (128-byte swizzle), completing on mbarriers.
//  * Warps 0-3 consume. Each owns a quarter of head_dim. QK: mma.sync
//    m16n8k16 with 16 keys as M and the query group as N (S^T = K Q^T), partial
//    over the warp's quarter; the four partials meet in shared memory (one
//    named barrier per tile), every warp forms the full scores of the tile,
//    runs the online softmax in fp32 (exp2 domain) and splits P into a bf16
//    high part and a bf16 remainder, both used as the B operand of PV:
//    O^T[d, h] += V^T[d, key] (P_hi + P_lo)^T[key, h] over its quarter.
//  * A unit whose tiles all fall in one CTA writes its normalised output
//    directly; units cut by a slice boundary leave (m, l, O) partials in the
//    workspace (slot = CTA + unit, which is unique because slices and units
//    are both contiguous in tile order). Each such CTA then takes a ticket on
//    the unit; the one that takes the last ticket combines all partials with
//    the log-sum-exp rule. No CTA ever waits for another.
//  * While a unit's last tile is in flight, the consumers load the next
//    unit's queries into registers.
//  * Rows of a partially visible page (before the window start or past the
//    end) are masked in the scores and their V rows zeroed in shared memory,
//    so stale or non-finite cache contents never reach the output.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace dec {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kChunkBytes = kBlockSize * 128;  // one TMA box: 16 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Two CTAs share each SM: every tile is 32 KB of K/V (2 pages of K and V, or
// 4 pages of K alone with k_eq_v at head_dim 256, ...), 3 tiles in flight per
// CTA, so each SM keeps two independent TMA pipelines and 8 consumer warps.
constexpr int kCtasPerSm = 2;
constexpr int kStageTarget = 32768;
constexpr int kInfoInts = 16;  // shared ints: warp sums, slice start, flags

// FP8 pages: the ring holds e4m3 tiles (half the bytes of a bf16 tile of the
// same keys) and their per-row scales; every consumer warp converts its own
// quarter of head_dim of a tile into a bf16 tile of the usual layout, which
// the unchanged QK / PV code then reads.
template <int HD, bool KEQV, bool FP8 = false>
struct Cfg {
  static constexpr int kChunks = HD / 64;
  static constexpr int kPageBytes = kChunks * kChunkBytes;
  static constexpr int kTilePages = kStageTarget / (kPageBytes * (KEQV ? 1 : 2));
  static constexpr int kTileKeys = kTilePages * kBlockSize;
  static constexpr int kSRow = kTileKeys < 32 ? 32 : kTileKeys;  // score-exchange row stride
  static constexpr int kKTileBytes = kTilePages * kPageBytes;
  static constexpr int kStageBytes = kKTileBytes * (KEQV ? 1 : 2);  // one bf16 tile
  static constexpr int kSRowF = kTileKeys < 32 ? 32 : kTileKeys;
  // FP8 tiles are half the size: four ring stages where two CTAs per SM still fit
  static constexpr int kStages =
      !FP8 ? 3
           : (1024 + 4 * (kStageBytes / 2) + kStageBytes + 4 * kTileKeys * 2 * 4 +
                  2 * kConsumerWarps * kQHeadsPerUnit * kSRowF * 4 + 64 + 64) *
                         kCtasPerSm <= 232448
                 ? 4
                 : 3;
  // e4m3 geometry: a TMA box is 16 rows x 64 one-byte codes
  static constexpr int kChunkBytes8 = kBlockSize * 64;
  static constexpr int kPageBytes8 = kChunks * kChunkBytes8;
  static constexpr int kKTileBytes8 = kTilePages * kPageBytes8;
  static constexpr int kRingStageBytes = FP8 ? kStageBytes / 2 : kStageBytes;
  static constexpr int kScaleFloats = kTileKeys * (KEQV ? 1 : 2);  // per ring stage
  static constexpr int kScaleBytes = FP8 ? kStages * kScaleFloats * 4 : 0;
  static constexpr int kConvBytes = FP8 ? kStageBytes : 0;
  static constexpr int kDPerWarp = HD / kConsumerWarps;
  static constexpr int kKSteps = kDPerWarp / 16;
  static constexpr int kMTiles = kDPerWarp / 16;
  static constexpr int kChunksPerWarp = kDPerWarp / 64;
  static constexpr int kSBufFloats = kConsumerWarps * kQHeadsPerUnit * kSRow;
  static constexpr int kTmaPerTile = kTilePages * kChunks * (KEQV ? 1 : 2);
  static constexpr int kSmemBytes = 1024 + kStages * kRingStageBytes + kConvBytes + kScaleBytes +
                                    2 * kSBufFloats * 4 + 2 * kStages * 8 + kInfoInts * 4;
  static_assert(kTilePages >= 1, "tile of at least one page");
  static_assert(kTmaPerTile <= 32, "one TMA box per producer lane");
  static_assert(kSmemBytes * kCtasPerSm <= 232448, "shared memory per SM");
};

// Eight e4m3 codes (8 bytes) as eight bf16 values (16 bytes). Every e4m3
// value has at most four significant bits and an exponent in [-9, 8], so it
// is exact in f16 and then in bf16 (the upper half of its float).
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 in) {
  uint32_t out[4];
  const uint32_t w[2] = {in.x, in.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t pair =
        static_cast<__nv_fp8x2_storage_t>((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
    const float lo = __half2float(__half(__half_raw{h.x}));
    const float hi = __half2float(__half(__half_raw{h.y}));
    out[i] = __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// XOR swizzle of the key index in the score-exchange buffer: conflict-free
// for both the fragment-layout writes and the row-wise float2 reads.
__device__ __forceinline__ int sbuf_key(int qh, int key) {
  return key ^ (((qh ^ (qh >> 2)) & 3) << 3);
}

// ---------------------------------------------------------------- sequences
// What one sequence contributes to the tile list, from its seq_len alone: the
// length after validation (negative -> 0, longer than the block-table row ->
// the row's capacity), the first visible position (only the last min(len, W)
// keys of a sliding layer) and the tiles of each of its units.
struct SeqInfo {
  int len, lo, ntu;
};
__device__ __forceinline__ SeqInfo seq_info(const int32_t* __restrict__ seq_lens, int s,
                                            int window, int cap, int tile_pages) {
  int len = seq_lens[s];
  len = len < 0 ? 0 : (len > cap ? cap : len);
  const int lo = (window > 0 && len > window) ? len - window : 0;
  int ntu = 0;
  if (len > 0) {
    const int npages = (len - 1) / kBlockSize - lo / kBlockSize + 1;
    ntu = (npages + tile_pages - 1) / tile_pages;
  }
  return SeqInfo{len, lo, ntu};
}

// ---------------------------------------------------------------- walker
// Iterates the global tile list in order: sequence, unit, tile. Sequence
// data comes straight from seq_lens; tile_off (the first tile of the current
// sequence) is carried along.
struct Walker {
  const int32_t* seq_lens;
  int n_seqs, ups, window, cap, tile_pages;
  int s, unit, tile;
  int ntu, len, lo, tile_off;

  __device__ void load_seq() {
    const SeqInfo i = seq_info(seq_lens, s, window, cap, tile_pages);
    len = i.len; lo = i.lo; ntu = i.ntu;
  }
  // s0 holds tile t and its first tile is off0
  __device__ void init(const int32_t* sl, int ns, int u, int win, int cp, int tp, int s0,
                       int off0, int t) {
    seq_lens = sl; n_seqs = ns; ups = u; window = win; cap = cp; tile_pages = tp;
    s = s0;
    tile_off = off0;
    load_seq();
    const int rem = t - tile_off;
    unit = ntu > 0 ? rem / ntu : 0;
    tile = rem - unit * ntu;
  }
  __device__ void advance() {
    if (++tile < ntu) return;
    tile = 0;
    if (++unit < ups) return;
    unit = 0;
    tile_off += ntu * ups;
    for (++s; s < n_seqs; ++s) {  // sequences without visible keys have no tiles
      load_seq();
      if (ntu > 0) break;
    }
  }
  __device__ int first_page() const { return lo / kBlockSize; }
  __device__ int last_page() const { return len > 0 ? (len - 1) / kBlockSize : -1; }
  __device__ int unit_first_tile() const { return tile_off + unit * ntu; }
  __device__ int global_unit() const { return s * ups + unit; }
};

// ---------------------------------------------------------------- merge
// Combines the partial results of unit u held by CTAs c0..c1 (slots c + u):
// M = max m_i, l = sum l_i 2^(m_i - M), out = sum O_i 2^(m_i - M) / l,
// lse = (M + log2 l) ln 2. Partials are read through L2 (written by other SMs).
template <int HD>
__device__ void merge_unit(int u, int c0, int c1, int nh, float* out_rows, float* lse_rows,
                           const float* ws_o, const float2* ws_ml, int tid, int nthreads) {
  for (int qh = 0; qh < nh; ++qh) {
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c)
      M = fmaxf(M, __ldcg(&ws_ml[(static_cast<int64_t>(c) + u) * kQHeadsPerUnit + qh].x));
    float Lsum = 0.f;
    for (int c = c0; c <= c1; ++c) {
      const float2 ml = __ldcg(&ws_ml[(static_cast<int64_t>(c) + u) * kQHeadsPerUnit + qh]);
      Lsum += ml.y * exp2f(ml.x - M);
    }
    const float inv = 1.f / Lsum;
    for (int d = tid; d < HD; d += nthreads) {
      float acc = 0.f;
      for (int c = c0; c <= c1; ++c) {
        const int64_t slot = static_cast<int64_t>(c) + u;
        const float wgt = exp2f(__ldcg(&ws_ml[slot * kQHeadsPerUnit + qh].x) - M);
        acc += __ldcg(&ws_o[(slot * kQHeadsPerUnit + qh) * HD + d]) * wgt;
      }
      out_rows[qh * HD + d] = acc * inv;
    }
    if (tid == 0 && lse_rows != nullptr) lse_rows[qh] = (M + log2f(Lsum)) * kLn2;
  }
}

// ---------------------------------------------------------------- split
template <int HD, bool KEQV, bool FP8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map,
                    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
                    int max_blocks, int64_t num_blocks, const int32_t* __restrict__ seq_lens,
                    int n_seqs, int n_q, int n_kv, int group, int qchunks, int window,
                    float scale, float softcap, float* __restrict__ out,
                    float* __restrict__ lse, float* __restrict__ ws_o,
                    float2* __restrict__ ws_ml, int32_t* __restrict__ tickets,
                    const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                    int32_t* err, int stall_cta, int stall_tile, AppendArgs append) {
  using C = Cfg<HD, KEQV, FP8>;
  constexpr int TP = C::kTilePages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;                                        // the ring
  uint8_t* conv = stages + C::kStages * C::kRingStageBytes;      // FP8: converted tile
  float* scales = reinterpret_cast<float*>(conv + C::kConvBytes);  // FP8: [stage][K/V][key]
  float* sbuf = scales + C::kScaleBytes / 4;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sbuf + 2 * C::kSBufFloats);
  uint64_t* empty_bar = full_bar + C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_bar + C::kStages);
  volatile int* cons_abort = abort_flag + 1;  // written only by consumer warps
  volatile int* merge_flag = abort_flag + 2;  // this CTA merges the current unit
  int* info = const_cast<int*>(abort_flag) + 4;  // warp sums [0, 5), slice start [5, 7)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      // FP8: the TMA bytes plus one arrival per producer lane for the scales
      mbar_init(&full_bar[i], FP8 ? 1 + 32 : 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    *abort_flag = 0;
    *cons_abort = 0;
    *merge_flag = 0;
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&k_map);
    if (!KEQV) prefetch_tensormap(&v_map);
  }
  __syncthreads();

  // ---- this CTA's slice of the global tile list. Every CTA forms the same
  // integer sums over seq_lens: thread i sums the tiles of a contiguous run of
  // sequences, a block scan gives the total and each run's first tile, and the
  // thread whose run holds the slice's first tile finds that sequence.
  const int ups = n_kv * qchunks;
  const int cap = max_blocks * kBlockSize;
  const int tid = threadIdx.x;
  const int run = (n_seqs + kThreads - 1) / kThreads;
  const int s_lo = min(n_seqs, tid * run), s_hi = min(n_seqs, s_lo + run);
  int mine = 0;
  for (int s = s_lo; s < s_hi; ++s) mine += seq_info(seq_lens, s, window, cap, TP).ntu * ups;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) info[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int i = 0; i < kConsumerWarps + 1; ++i) {
    if (i < warp) before += info[i];
    total += info[i];
  }
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int t_begin = blockIdx.x * per;
  const int t_end = min(total, t_begin + per);
  {
    int off = before + incl - mine;
    if (t_begin < t_end && off <= t_begin && t_begin < off + mine) {
      for (int s = s_lo; s < s_hi; ++s) {
        const int tl = seq_info(seq_lens, s, window, cap, TP).ntu * ups;
        if (t_begin < off + tl) {
          info[5] = s;
          info[6] = off;
          break;
        }
        off += tl;
      }
    }
  }
  // Sequences without a visible key have no tiles: CTA s mod grid writes their
  // zero rows and lse = -inf, and flags invalid lengths of its sequences.
  for (int s = blockIdx.x; s < n_seqs; s += gridDim.x) {
    const int raw = seq_lens[s];
    if (tid == 0 && raw < 0) flag_error(err, PSW_DEVERR_LENGTH);
    if (tid == 0 && raw > cap) flag_error(err, PSW_DEVERR_CAPACITY);
    if (raw <= 0) {
      float4* row = reinterpret_cast<float4*>(out + static_cast<int64_t>(s) * n_q * HD);
      for (int i = tid; i < n_q * HD / 4; i += kThreads) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lse != nullptr)
        for (int i = tid; i < n_q; i += kThreads) lse[static_cast<int64_t>(s) * n_q + i] = -INFINITY;
    }
  }
  __syncthreads();
  if (t_begin >= t_end) return;
  const int start_seq = info[5], start_off = info[6];

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    Walker w;
    w.init(seq_lens, n_seqs, ups, window, cap, TP, start_seq, start_off, t_begin);
    // lane -> (K/V, page in tile, chunk) of its TMA box
    const int which = lane / (TP * C::kChunks);
    const int lp = (lane % (TP * C::kChunks)) / C::kChunks;
    const int lc = lane % C::kChunks;
    int issued = 0;
    for (int t = t_begin; t < t_end; ++t, ++issued) {
      // testing hook: this copy is never issued, so a consumer wait runs out
      if (static_cast<int>(blockIdx.x) == stall_cta && issued == stall_tile) break;
      const int stage = issued % C::kStages;
      const uint32_t ph = (issued / C::kStages) & 1;
      const int kvh = w.unit / qchunks;
      const int page0 = w.first_page() + w.tile * TP;
      const int npages = min(TP, w.last_page() - page0 + 1);
      int blk = -1;
      if (lane < npages) {
        // the table row is read only inside [0, max_blocks), whatever the walk
        // says (it stays there by construction: last_page < max_blocks)
        const int page = page0 + lane;
        if (page < 0 || page >= max_blocks) {
          flag_error(err, PSW_DEVERR_CAPACITY);
        } else {
          blk = block_table[static_cast<int64_t>(w.s) * max_blocks + page];
          if (blk < 0 || blk >= num_blocks) {
            flag_error(err, PSW_DEVERR_BLOCK_ID);
            blk = -1;  // out-of-range box: TMA fills zeros
          }
        }
      }
      const int my_blk = __shfl_sync(0xffffffffu, blk, lp);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty_bar[stage], ph ^ 1);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag) {
        if (lane == 0) { flag_error(err, PSW_DEVERR_PIPELINE); *abort_flag = 1; }
        break;
      }
      if (lane == 0)
        mbar_arrive_expect_tx(
            &full_bar[stage],
            static_cast<uint32_t>(npages * (FP8 ? C::kPageBytes8 : C::kPageBytes) *
                                  (KEQV ? 1 : 2)));
      __syncwarp();
      if (lane < C::kTmaPerTile && lp < npages) {
        uint8_t* dst =
            FP8 ? stages + stage * C::kRingStageBytes + which * C::kKTileBytes8 +
                      lp * C::kPageBytes8 + lc * C::kChunkBytes8
                : stages + stage * C::kStageBytes + which * C::kKTileBytes + lp * C::kPageBytes +
                      lc * kChunkBytes;
        const CUtensorMap* map = (which == 0) ? &k_map : &v_map;
        tma_load_3d_hint(dst, map, &full_bar[stage], 0, kvh * C::kChunks + lc,
                         my_blk * kBlockSize, policy);
      }
      if constexpr (FP8) {
        // the tile's row scales: key i of the tile from page i / 16, row i % 16
        // (0 for pages past the sequence end or with a bad block id)
        float* sc = scales + stage * C::kScaleFloats;
#pragma unroll
        for (int i0 = 0; i0 < C::kTileKeys; i0 += 32) {
          const int i = i0 + lane;
          const int pblk = __shfl_sync(0xffffffffu, blk, (i / kBlockSize) % 32);
          float ks = 0.f, vs = 0.f;
          if (i < C::kTileKeys && i / kBlockSize < npages && pblk >= 0) {
            const int64_t r =
                (static_cast<int64_t>(pblk) * kBlockSize + i % kBlockSize) * n_kv + kvh;
            ks = k_scale[r];
            if (!KEQV) vs = v_scale[r];
          }
          if (i < C::kTileKeys) {
            sc[i] = ks;
            if (!KEQV) sc[C::kTileKeys + i] = vs;
          }
        }
        mbar_arrive(&full_bar[stage]);  // every lane: its scale stores are released
      }
      w.advance();
    }
    // drain: the last phase of every stage used must have landed before exit
    if (lane == 0) {
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(&full_bar[i % C::kStages], (i / C::kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t4 = lane & 3;
  const float scale_l2 = scale * kLog2e;
  const bool use_cap = softcap > 0.f;
  float o[C::kMTiles][4];
  uint32_t qf[C::kKSteps][2], qn[C::kKSteps][2];
  float m_run = -INFINITY, l_run = 0.f;
  int nh = 0, hb = 0;
  bool have_next = false;
  // Q fragments (B operand of QK) of unit `unit` of sequence `sq` for this lane
  auto load_q = [&](int sq, int unit, uint32_t (&dst)[C::kKSteps][2]) {
    const int kvh = unit / qchunks, qc = unit - kvh * qchunks;
    const int hb_u = kvh * group + qc * kQHeadsPerUnit;
    const int nh_u = min(kQHeadsPerUnit, group - qc * kQHeadsPerUnit);
    const __nv_bfloat16* qrow =
        q + (static_cast<int64_t>(sq) * n_q + hb_u + g) * HD + warp * C::kDPerWarp + t4 * 2;
    #pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
      if (g < nh_u) {
        dst[ks][0] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16));
        dst[ks][1] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 8));
      } else {
        dst[ks][0] = 0u;
        dst[ks][1] = 0u;
      }
    }
  };

  // per-lane ldmatrix geometry
  const int j8 = lane >> 3, r8 = lane & 7;
  const int qk_row = (j8 & 1) * 8 + r8;       // key row within a page (QK, A = K)
  const int qk_unit_add = j8 >> 1;            // +8 columns of d
  const int pv_row = (j8 >> 1) * 8 + r8;      // key row within a page (PV, A = V^T)
  const int pv_dadd = (j8 & 1) * 8;
  const uint32_t stages_u32 = smem_u32(stages);

  Walker w;
  w.init(seq_lens, n_seqs, ups, window, cap, TP, start_seq, start_off, t_begin);
  int consumed = 0;
  for (int t = t_begin; t < t_end; ++t, ++consumed) {
    const int stage = consumed % C::kStages;
    const uint32_t ph = (consumed / C::kStages) & 1;
    const bool unit_start = (w.tile == 0) || (t == t_begin);
    if (unit_start) {
      const int kvh = w.unit / qchunks, qc = w.unit - (w.unit / qchunks) * qchunks;
      hb = kvh * group + qc * kQHeadsPerUnit;
      nh = min(kQHeadsPerUnit, group - qc * kQHeadsPerUnit);
      if (have_next) {
        #pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) { qf[ks][0] = qn[ks][0]; qf[ks][1] = qn[ks][1]; }
      } else {
        load_q(w.s, w.unit, qf);
      }
      // prefetch the next unit's Q (if this CTA reaches it) while this one runs
      Walker nx = w;
      nx.tile = nx.ntu - 1;
      nx.advance();
      have_next = nx.s < n_seqs && nx.unit_first_tile() < t_end;
      if (have_next) load_q(nx.s, nx.unit, qn);
      #pragma unroll
      for (int i = 0; i < C::kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }
    const int page0 = w.first_page() + w.tile * TP;
    const int npages = min(TP, w.last_page() - page0 + 1);
    const int pos0 = page0 * kBlockSize;

    // A timed-out wait is decided collectively after the named barrier below,
    // so that all consumer warps pass the same number of barriers.
    const bool landed = mbar_wait(&full_bar[stage], ph);
    if (!landed && lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *cons_abort = 1;
    }
    // Append mode: this unit's last tile holds the step's new token
    // (position len - 1); its K/V rows come from the inputs into this warp's
    // chunks of the staged tile (each warp reads only its own chunks), and
    // the unit of the first query chunk also stores them in the pools for
    // later steps. A bad block id or length was flagged by the producer or
    // the prologue; such a row is left alone.
    if constexpr (!FP8) {
      if (append.k_new != nullptr && landed && w.tile == w.ntu - 1 && w.len > 0 &&
          seq_lens[w.s] == w.len) {
        const int pos = w.len - 1, page = pos / kBlockSize, row = pos % kBlockSize;
        const int kk = page - page0;
        const int kvh = w.unit / qchunks;
        const int32_t blk = page < max_blocks
                                ? block_table[static_cast<int64_t>(w.s) * max_blocks + page]
                                : -1;
        if (blk >= 0 && blk < num_blocks) {
          const bool to_pool = w.unit == kvh * qchunks;
          constexpr int kUnits = C::kChunksPerWarp * 8;  // 16-byte units of this warp's dims
          uint8_t* tile = stages + stage * C::kStageBytes + kk * C::kPageBytes;
          const int64_t slot = static_cast<int64_t>(blk) * kBlockSize + row;
          for (int idx = lane; idx < (KEQV ? 1 : 2) * kUnits; idx += 32) {
            const int which = idx / kUnits, rem = idx - which * kUnits;
            const int c = warp * C::kChunksPerWarp + rem / 8, u = rem & 7;
            const int d = c * 64 + u * 8;
            const uint4 val = *reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(which ? append.v_new : append.k_new) +
                (static_cast<int64_t>(w.s) * n_kv + kvh) * HD + d);
            *reinterpret_cast<uint4*>(tile + which * C::kKTileBytes + c * kChunkBytes + row * 128 +
                                      ((u ^ (row & 7)) << 4)) = val;
            if (to_pool)
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which ? append.v_pool
                                                                           : append.k_pool) +
                                        (slot * n_kv + kvh) * HD + d) = val;
          }
          fence_proxy_async_smem();  // the stage is later refilled by TMA
          __syncwarp();
        }
      }
    }
    // FP8: this warp converts its quarter of head_dim of the tile (K, and V
    // unless k_eq_v) into the bf16 tile, keeps the scales of its keys (same
    // order as the scores below) and releases the ring stage at once
    float ksc[TP][4], vsc[TP][4];
    if constexpr (FP8) {
      if (landed) {
        const uint8_t* ring = stages + stage * C::kRingStageBytes;
#pragma unroll
        for (int which = 0; which < (KEQV ? 1 : 2); ++which) {
#pragma unroll
          for (int pg = 0; pg < TP; ++pg) {
#pragma unroll
            for (int cw = 0; cw < C::kChunksPerWarp; ++cw) {
              const int c = warp * C::kChunksPerWarp + cw;
              const uint8_t* src =
                  ring + which * C::kKTileBytes8 + pg * C::kPageBytes8 + c * C::kChunkBytes8;
              uint8_t* dst = conv + which * C::kKTileBytes + pg * C::kPageBytes + c * kChunkBytes;
#pragma unroll
              for (int idx = lane; idx < kBlockSize * 8; idx += 32) {
                const int row = idx >> 3, u = idx & 7;  // 8 codes -> one 16-byte bf16 unit
                const uint2 in = *reinterpret_cast<const uint2*>(src + row * 64 + u * 8);
                *reinterpret_cast<uint4*>(dst + row * 128 + ((u ^ (row & 7)) << 4)) =
                    e4m3x8_to_bf16x8(in);
              }
            }
          }
        }
        const float* sc = scales + stage * C::kScaleFloats;
#pragma unroll
        for (int kk = 0; kk < TP; ++kk)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = kk * 16 + (e >> 1) * 8 + 2 * t4 + (e & 1);
            ksc[kk][e] = sc[key];
            vsc[kk][e] = KEQV ? ksc[kk][e] : sc[C::kTileKeys + key];
          }
        __syncwarp();  // the warp's ldmatrix reads what its lanes converted
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
      }
    }
    const uint32_t kbase = FP8 ? smem_u32(conv) : stages_u32 + stage * C::kStageBytes;
    const uint32_t vbase = KEQV ? kbase : kbase + C::kKTileBytes;

    // ---- QK over this warp's quarter of head_dim: S^T[key, qh]. Even and
    // odd head_dim steps go to two accumulators (two independent MMA chains
    // per page instead of one), added at the end.
    float sacc[TP][4];
    if (landed) {
      float sacc2[TP][4];
      #pragma unroll
      for (int mt = 0; mt < TP; ++mt) {
        #pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][e] = sacc2[mt][e] = 0.f;
        #pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
          const int d0 = warp * C::kDPerWarp + ks * 16;
          const int c = d0 >> 6;
          const int u = ((d0 & 63) >> 3) + qk_unit_add;
          const uint32_t addr = kbase + mt * C::kPageBytes + c * kChunkBytes + qk_row * 128 +
                                ((u ^ (qk_row & 7)) << 4);
          uint32_t a[4];
          ldsm_x4(addr, a);
          mma_bf16_16816((ks & 1) ? sacc2[mt] : sacc[mt], a, qf[ks][0], qf[ks][1]);
        }
        #pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][e] += sacc2[mt][e];
      }
    } else {
      #pragma unroll
      for (int mt = 0; mt < TP; ++mt) sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
    }
    float* sb = sbuf + (consumed & 1) * C::kSBufFloats;
    {
      float* mine = sb + warp * kQHeadsPerUnit * C::kSRow;
      #pragma unroll
      for (int mt = 0; mt < TP; ++mt) {
        const int k0 = mt * 16 + g;
        const int qa = 2 * t4, qb = 2 * t4 + 1;
        mine[qa * C::kSRow + sbuf_key(qa, k0)] = sacc[mt][0];
        mine[qb * C::kSRow + sbuf_key(qb, k0)] = sacc[mt][1];
        mine[qa * C::kSRow + sbuf_key(qa, k0 + 8)] = sacc[mt][2];
        mine[qb * C::kSRow + sbuf_key(qb, k0 + 8)] = sacc[mt][3];
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
    if (*cons_abort) {
      if (lane == 0) *abort_flag = 1;  // stops the producer at its next tile
      break;
    }

    // ---- full scores for qh = g, keys kk*16 + 2*t4 + {0, 1, 8, 9}
    float sv[TP][4];
    float mx = -INFINITY;
    #pragma unroll
    for (int kk = 0; kk < TP; ++kk) {
      #pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kk * 16 + e * 8 + 2 * t4;
        float2 acc = make_float2(0.f, 0.f);
        #pragma unroll
        for (int ww = 0; ww < kConsumerWarps; ++ww) {
          const float2 v2 = *reinterpret_cast<const float2*>(
              sb + (ww * kQHeadsPerUnit + g) * C::kSRow + sbuf_key(g, key));
          acc.x += v2.x;
          acc.y += v2.y;
        }
        float x0 = acc.x, x1 = acc.y;
        if constexpr (FP8) {  // the key's row scale
          x0 *= ksc[kk][2 * e];
          x1 *= ksc[kk][2 * e + 1];
        }
        if (use_cap) {
          x0 = softcap * tanhf(x0 * scale / softcap) * kLog2e;
          x1 = softcap * tanhf(x1 * scale / softcap) * kLog2e;
        } else {
          x0 *= scale_l2;
          x1 *= scale_l2;
        }
        const int p0 = pos0 + key;
        if (p0 < w.lo || p0 >= w.len) x0 = -INFINITY;
        if (p0 + 1 < w.lo || p0 + 1 >= w.len) x1 = -INFINITY;
        sv[kk][2 * e] = x0;
        sv[kk][2 * e + 1] = x1;
        mx = fmaxf(mx, fmaxf(x0, x1));
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);  // finite: every tile holds a visible key
    const float alpha = exp2f(m_run - m_new);
    // P = P_hi + P_lo, both bf16: the PV product then carries P to ~2^-17
    // relative instead of bf16's 2^-9.
    uint32_t pf[TP][2], pl[TP][2];
    float psum = 0.f;
    #pragma unroll
    for (int kk = 0; kk < TP; ++kk) {
      float p0 = exp2f(sv[kk][0] - m_new), p1 = exp2f(sv[kk][1] - m_new);
      float p2 = exp2f(sv[kk][2] - m_new), p3 = exp2f(sv[kk][3] - m_new);
      psum += (p0 + p1) + (p2 + p3);
      if constexpr (FP8) {  // the V row scale folded into P (masked keys stay 0)
        p0 = p0 > 0.f ? p0 * vsc[kk][0] : 0.f;
        p1 = p1 > 0.f ? p1 * vsc[kk][1] : 0.f;
        p2 = p2 > 0.f ? p2 * vsc[kk][2] : 0.f;
        p3 = p3 > 0.f ? p3 * vsc[kk][3] : 0.f;
      }
      pf[kk][0] = pack_bf16x2(p0, p1);
      pf[kk][1] = pack_bf16x2(p2, p3);
      const float2 h0 = unpack_bf16x2(pf[kk][0]), h1 = unpack_bf16x2(pf[kk][1]);
      pl[kk][0] = pack_bf16x2(p0 - h0.x, p1 - h0.y);
      pl[kk][1] = pack_bf16x2(p2 - h1.x, p3 - h1.y);
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;

    // ---- zero the V rows of partially visible pages (this warp's chunks)
    #pragma unroll
    for (int kk = 0; kk < TP; ++kk) {
      const int pf_pos = pos0 + kk * kBlockSize;
      const int r_lo = max(0, w.lo - pf_pos);
      const int r_hi = min(kBlockSize, w.len - pf_pos);
      if (kk < npages && (r_lo > 0 || r_hi < kBlockSize)) {
        uint8_t* vpage = (FP8 ? conv : stages + stage * C::kStageBytes) +
                         (KEQV ? 0 : C::kKTileBytes) + kk * C::kPageBytes;
        for (int idx = lane; idx < kBlockSize * 8 * C::kChunksPerWarp; idx += 32) {
          const int row = idx / (8 * C::kChunksPerWarp);
          const int rem = idx - row * (8 * C::kChunksPerWarp);
          const int c = warp * C::kChunksPerWarp + rem / 8;
          const int u = rem & 7;
          if (row < r_lo || row >= r_hi)
            *reinterpret_cast<uint4*>(vpage + c * kChunkBytes + row * 128 + u * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    }

    // ---- rescale O^T (only when some query head's maximum rose: alpha is
    // exactly 1 otherwise) and accumulate PV over this warp's quarter
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
      const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * t4) * 4);
      const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * t4 + 1) * 4);
      #pragma unroll
      for (int mt2 = 0; mt2 < C::kMTiles; ++mt2) {
        o[mt2][0] *= a0;
        o[mt2][1] *= a1;
        o[mt2][2] *= a0;
        o[mt2][3] *= a1;
      }
    }
    #pragma unroll
    for (int kk = 0; kk < TP; ++kk) {
      if (kk < npages) {
        #pragma unroll
        for (int mt2 = 0; mt2 < C::kMTiles; ++mt2) {
          const int d = warp * C::kDPerWarp + mt2 * 16 + pv_dadd;
          const int c = d >> 6;
          const int u = (d & 63) >> 3;
          const uint32_t addr = vbase + kk * C::kPageBytes + c * kChunkBytes + pv_row * 128 +
                                ((u ^ (pv_row & 7)) << 4);
          uint32_t a[4];
          ldsm_x4_trans(addr, a);
          mma_bf16_16816(o[mt2], a, pf[kk][0], pf[kk][1]);
          mma_bf16_16816(o[mt2], a, pl[kk][0], pl[kk][1]);
        }
      }
    }
    __syncwarp();
    if (!FP8 && lane == 0) mbar_arrive(&empty_bar[stage]);

    // ---- end of this CTA's share of the unit: write the result or a partial
    const bool unit_end = (w.tile == w.ntu - 1) || (t == t_end - 1);
    if (unit_end) {
      float l_tot = l_run;
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
      l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
      const int uf = w.unit_first_tile();
      const bool complete = uf >= t_begin && uf + w.ntu - 1 < t_end;
      const int64_t slot = static_cast<int64_t>(blockIdx.x) + w.global_unit();
      #pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int qh = 2 * t4 + e;
        const float lq = __shfl_sync(0xffffffffu, l_tot, qh * 4);
        if (qh < nh) {
          const float inv = 1.f / lq;
          #pragma unroll
          for (int mt2 = 0; mt2 < C::kMTiles; ++mt2) {
            const int d = warp * C::kDPerWarp + mt2 * 16 + g;
            if (complete) {
              float* orow = out + (static_cast<int64_t>(w.s) * n_q + hb + qh) * HD;
              orow[d] = o[mt2][e] * inv;
              orow[d + 8] = o[mt2][2 + e] * inv;
            } else {
              float* prow = ws_o + (slot * kQHeadsPerUnit + qh) * HD;
              prow[d] = o[mt2][e];
              prow[d + 8] = o[mt2][2 + e];
            }
          }
        }
      }
      if (warp == 0 && t4 == 0 && g < nh) {
        if (complete) {
          if (lse != nullptr)
            lse[static_cast<int64_t>(w.s) * n_q + hb + g] = (m_run + log2f(l_tot)) * kLn2;
        } else {
          ws_ml[slot * kQHeadsPerUnit + g] = make_float2(m_run, l_tot);
        }
      }
      if (!complete) {
        // The CTA that finishes a unit's last segment merges all segments:
        // each CTA publishes its partial, then takes a ticket; nobody waits.
        // The ticket of a cut unit lives at its first CTA c0 (a CTA starts at
        // most one cut unit: its last), and the merging CTA, the last to touch
        // it in this call, sets it back to zero for the next call.
        const int u = w.global_unit();
        const int c0 = uf / per, c1 = (uf + w.ntu - 1) / per;
        __threadfence();
        named_bar_sync(1, kConsumerWarps * 32);
        if (threadIdx.x == 0) {
          const bool last = atomicAdd(&tickets[c0], 1) == c1 - c0;
          if (last) atomicExch(&tickets[c0], 0);
          *merge_flag = last;
        }
        named_bar_sync(1, kConsumerWarps * 32);
        if (*merge_flag) {
          __threadfence();
          merge_unit<HD>(u, c0, c1, nh, out + (static_cast<int64_t>(w.s) * n_q + hb) * HD,
                         lse == nullptr ? nullptr : lse + static_cast<int64_t>(w.s) * n_q + hb,
                         ws_o, ws_ml, threadIdx.x, kConsumerWarps * 32);
        }
      }
    }
    w.advance();
  }
}

template <int HD, bool KEQV, bool FP8>
int launch(const LayerArgs& L, const void* q, const CUtensorMap& k_map, const CUtensorMap& v_map,
           const int32_t* block_table, int max_blocks, int64_t num_blocks, const int32_t* seq_lens,
           int n_seqs, float* out, float* lse, void* ws, size_t ws_bytes, int num_sms,
           int32_t* err, cudaStream_t stream, const float* k_scale, const float* v_scale,
           AppendArgs append) {
  using C = Cfg<HD, KEQV, FP8>;
  const int grid = num_sms * kCtasPerSm < kMaxDecodeCtas ? num_sms * kCtasPerSm : kMaxDecodeCtas;
  const DecodeWorkspace lay = decode_workspace_layout(L, n_seqs, kMaxDecodeCtas);
  if (ws_bytes < lay.total) return PSW_EWORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* ws_o = reinterpret_cast<float*>(base + lay.o_offset);
  float2* ws_ml = reinterpret_cast<float2*>(base + lay.ml_offset);
  int32_t* tickets = reinterpret_cast<int32_t*>(base + lay.ticket_offset);
  if (set_smem_limit(reinterpret_cast<const void*>(decode_split_kernel<HD, KEQV, FP8>),
                     C::kSmemBytes) != PSW_OK)
    return PSW_ELAUNCH;
  const StallHook stall = stall_hook(kStallDecode);
  decode_split_kernel<HD, KEQV, FP8><<<grid, kThreads, C::kSmemBytes, stream>>>(
      k_map, v_map, static_cast<const __nv_bfloat16*>(q), block_table, max_blocks, num_blocks,
      seq_lens, n_seqs, L.n_q, L.n_kv, L.group(), L.qchunks(), L.window, L.scale, L.softcap,
      out, lse, ws_o, ws_ml, tickets, k_scale, v_scale, err, stall.cta, stall.tile, append);
  return cudaGetLastError() == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace dec

DecodeWorkspace decode_workspace_layout(const LayerArgs& L, int n_seqs, int max_ctas) {
  DecodeWorkspace w{};
  auto align = [](size_t x) { return (x + kDecodePlanAlign - 1) / kDecodePlanAlign * kDecodePlanAlign; };
  const size_t slots = static_cast<size_t>(max_ctas) +
                       static_cast<size_t>(n_seqs) * L.n_kv * L.qchunks();
  // merge tickets, one per CTA, in the zero-kept counter block at the start
  w.ticket_offset = 0;
  w.ticket_bytes = kWsCounterBytes;
  w.o_bytes = align(slots * kQHeadsPerUnit * L.hd * sizeof(float));
  w.ml_bytes = align(slots * kQHeadsPerUnit * sizeof(float2));
  w.o_offset = kWsCounterBytes;
  w.ml_offset = w.o_offset + w.o_bytes;
  w.total = w.ml_offset + w.ml_bytes;
  return w;
}

int launch_decode(const LayerArgs& L, const void* q, const CUtensorMap& k_map,
                  const CUtensorMap& v_map, const int32_t* block_table, int max_blocks,
                  int64_t num_blocks, const int32_t* seq_lens, int n_seqs, float* out, float* lse,
                  void* ws, size_t ws_bytes, int num_sms, int32_t* err, cudaStream_t stream,
                  const float* k_scale, const float* v_scale, AppendArgs append) {
  if (n_seqs == 0) return PSW_OK;
  const bool fp8 = k_scale != nullptr;
#define PSW_DEC(HD, KV, F8)                                                                  \
  dec::launch<HD, KV, F8>(L, q, k_map, v_map, block_table, max_blocks, num_blocks, seq_lens, \
                          n_seqs, out, lse, ws, ws_bytes, num_sms, err, stream, k_scale, v_scale, \
                          append)
  if (L.hd == 256) {
    if (fp8) return L.k_eq_v ? PSW_DEC(256, true, true) : PSW_DEC(256, false, true);
    return L.k_eq_v ? PSW_DEC(256, true, false) : PSW_DEC(256, false, false);
  }
  if (fp8) return L.k_eq_v ? PSW_DEC(512, true, true) : PSW_DEC(512, false, true);
  return L.k_eq_v ? PSW_DEC(512, true, false) : PSW_DEC(512, false, false);
#undef PSW_DEC
}

}  // namespace psw
