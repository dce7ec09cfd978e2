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
//  * Warp 4 (producer) streams K and V tiles of BN keys (64 for head_dim 256,
//    32 for 512) into a 2-stage ring, one 2 KB TMA box per (page, 64-column
//    chunk). Pages past the sequence end load as zeros (out-of-range box).
//  * Warp 5 (one elected thread) issues tcgen05.mma: S = Q K^T (SS, both
//    K-major) into TMEM, and O += P V (TS: P from TMEM, V MN-major from shared
//    memory). QK of tile j+1 is issued before PV of tile j so the tensor pipe
//    works while the softmax warps run.
//  * Warps 0-3 (one thread per row) read S from TMEM, apply scale, softcap and
//    the band/causal predicate, run the online softmax in fp32 (exp2 domain,
//    lazy rescaling of O only when the running max grows by more than 2^8),
//    and write P back to TMEM as a bf16 high part and a bf16 remainder; both
//    are multiplied into O, so P enters the product to about 2^-17 relative.
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

constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kRows = 128;
constexpr int kPageBoxBytes = kBlockSize * 128;  // one TMA box: 16 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int HD, bool KEQV>
struct Cfg {
  static constexpr int kQChunks = HD / 64;
  static constexpr int kBN = (HD == 256) ? 64 : 32;
  static constexpr int kPagesPerTile = kBN / kBlockSize;
  static constexpr int kOCols = 256;
  static constexpr int kDSplit = HD / kOCols;
  static constexpr int kVChunks = kOCols / 64;
  static constexpr int kQBytes = kQChunks * kRows * 128;
  static constexpr int kChunkTileBytes = kBN * 128;  // one 64-column chunk of a K/V tile
  static constexpr int kKBytes = kQChunks * kChunkTileBytes;
  static constexpr int kVBytes = KEQV ? 0 : kVChunks * kChunkTileBytes;
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kStages = 2;
  static constexpr int kSmemBytes = 1024 + kQBytes + kStages * kStageBytes + 256;
  static constexpr int kTmemO = 0;
  static constexpr int kTmemS = 256;
  static constexpr int kTmemPhi = 256 + kBN;
  static constexpr int kTmemPlo = 256 + kBN + kBN / 2;
  static constexpr int kTmemCols = 512;
  static constexpr int kTmaPerStage = kPagesPerTile * (kQChunks + (KEQV ? 0 : kVChunks));
  static_assert(kTmaPerStage <= 32, "one TMA box per producer lane");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kTmemPlo + kBN / 2 <= kTmemCols, "tensor memory columns");
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full, s_free, p_full, pv_done, mma_drained;
  uint32_t tmem_base;
  int abort;     // set by any warp; read by the producer and the MMA issuer
  int sm_abort;  // set only by softmax threads, read after their named barrier
};

// softcap: cap * tanh(x / cap) with tanh from one exp2 and one reciprocal.
__device__ __forceinline__ float softcap_tanh(float x, float cap, float inv_cap) {
  const float y = x * inv_cap;
  const float t = exp2f(-2.f * kLog2e * fabsf(y));      // e^{-2|y|}
  const float th = __fdividef(1.f - t, 1.f + t);         // tanh |y|
  return cap * copysignf(th, y);
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
  uint8_t* stages = smem + C::kQBytes;
  Bars* bars = reinterpret_cast<Bars*>(stages + C::kStages * C::kStageBytes);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, kSoftmaxWarps);
    mbar_init(&bars->p_full, kSoftmaxWarps);
    mbar_init(&bars->pv_done, 1);
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&q_map);
      prefetch_tensormap(&k_map);
      if (!KEQV) prefetch_tensormap(&v_map);
      mbar_arrive_expect_tx(&bars->q_full,
                            static_cast<uint32_t>(C::kQChunks * group * T * 128));
      for (int c = 0; c < C::kQChunks; ++c)
        tma_load_3d(q_smem + c * (kRows * 128), &q_map, &bars->q_full, c * 64, kvh * group,
                    q0 + i0);
    }
    // lane -> (page in tile, chunk, K or V)
    const int per_page = C::kQChunks + (KEQV ? 0 : C::kVChunks);
    const int lp = lane / per_page;
    const int lc = lane - lp * per_page;
    const bool is_v = lc >= C::kQChunks;
    int issued = 0;
    for (int j = 0; j < nkt; ++j, ++issued) {
      const int stage = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      const int page0 = (kt0 + j) * C::kPagesPerTile;
      int blk = -1;
      if (lane < C::kPagesPerTile) {
        const int page = page0 + lane;
        if (page <= last_page) {
          blk = block_table[static_cast<int64_t>(b) * max_blocks + page];
          if (blk < 0 || blk >= num_blocks) {
            flag_error(err, PSW_DEVERR_BLOCK_ID);
            blk = -1;
          }
        }
      }
      const int my_blk = __shfl_sync(0xffffffffu, blk, lp < C::kPagesPerTile ? lp : 0);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&bars->kv_empty[stage], ph ^ 1);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag) {
        if (lane == 0) { flag_error(err, PSW_DEVERR_PIPELINE); *abort_flag = 1; }
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars->kv_full[stage], C::kStageBytes);
      __syncwarp();
      if (lane < C::kTmaPerStage) {
        uint8_t* st = stages + stage * C::kStageBytes;
        if (!is_v) {
          tma_load_3d(st + lc * C::kChunkTileBytes + lp * kPageBoxBytes, &k_map,
                      &bars->kv_full[stage], 0, kvh * C::kQChunks + lc, my_blk * kBlockSize);
        } else {
          const int cv = lc - C::kQChunks;
          tma_load_3d(st + C::kKBytes + cv * C::kChunkTileBytes + lp * kPageBoxBytes, &v_map,
                      &bars->kv_full[stage], 0, kvh * C::kQChunks + dh * C::kVChunks + cv,
                      my_blk * kBlockSize);
        }
      }
    }
    if (lane == 0) {  // drain this CTA's own copies before anyone leaves
      mbar_wait(&bars->q_full, 0);
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(&bars->kv_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_bf16_f32(kRows, BN, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(kRows, C::kOCols, 0, 1);
      const uint32_t q_base = smem_u32(q_smem);
      const uint32_t st_base = smem_u32(stages);
      bool ok = mbar_wait(&bars->q_full, 0);
      auto issue_pv = [&](int jj) {
        const uint32_t kb = st_base + (jj & 1) * C::kStageBytes;
        const uint32_t vb = KEQV ? kb + dh * C::kVChunks * C::kChunkTileBytes : kb + C::kKBytes;
        #pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t bdesc = tc::smem_desc(vb + ks * 16 * 128, C::kChunkTileBytes, 1024,
                                               tc::kSwizzle128B);
          tc::mma_ts(tmem + C::kTmemO, tmem + C::kTmemPhi + ks * 8, bdesc, idesc_pv,
                     (jj > 0 || ks > 0) ? 1u : 0u);
          tc::mma_ts(tmem + C::kTmemO, tmem + C::kTmemPlo + ks * 8, bdesc, idesc_pv, 1u);
        }
        tc::commit(&bars->pv_done);
        tc::commit(&bars->kv_empty[jj & 1]);
      };
      int j = 0;
      for (; ok && j < nkt; ++j) {
        ok = mbar_wait(&bars->kv_full[j & 1], (j >> 1) & 1);
        if (ok && j > 0) ok = mbar_wait(&bars->s_free, (j - 1) & 1);
        if (!ok || *abort_flag) break;
        tc::fence_after();
        const uint32_t kb = st_base + (j & 1) * C::kStageBytes;
        #pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const int c = ks >> 2;
          const uint64_t adesc = tc::smem_desc(q_base + c * (kRows * 128) + (ks & 3) * 32, 16,
                                               1024, tc::kSwizzle128B);
          const uint64_t bdesc = tc::smem_desc(kb + c * C::kChunkTileBytes + (ks & 3) * 32, 16,
                                               1024, tc::kSwizzle128B);
          tc::mma_ss(tmem + C::kTmemS, adesc, bdesc, idesc_qk, ks > 0 ? 1u : 0u);
        }
        tc::commit(&bars->s_full);
        if (j > 0) {
          ok = mbar_wait(&bars->p_full, (j - 1) & 1);
          if (!ok || *abort_flag) break;
          tc::fence_after();
          issue_pv(j - 1);
        }
      }
      if (ok && j == nkt && !*abort_flag) {
        ok = mbar_wait(&bars->p_full, (nkt - 1) & 1);
        if (ok) {
          tc::fence_after();
          issue_pv(nkt - 1);
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
    const int r = warp * 32 + lane;
    const int t = r / group;
    const int h = r - t * group;
    const bool row_ok = (t < tok_valid) && (r < group * T);
    const int p = past + i0 + t;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kTmemS;
    const uint32_t t_o = tmem + lane_off + C::kTmemO;
    const bool use_cap = softcap > 0.f;
    const float inv_cap = use_cap ? 1.f / softcap : 0.f;
    const float scale_l2 = scale * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    volatile int* sm_abort = &bars->sm_abort;  // written only by softmax threads
    for (int j = 0; j < nkt; ++j) {
      // every decision below is warp-uniform; the abort decision is taken by all
      // four softmax warps together after the named barrier
      bool okw = __all_sync(0xffffffffu, mbar_wait(&bars->s_full, j & 1));
      float x[BN];
      const int key0 = (kt0 + j) * BN;
      float alpha = 1.f;
      if (okw) {
        tc::fence_after();
        #pragma unroll
        for (int c16 = 0; c16 < BN / 16; ++c16) {
          uint32_t v[16];
          tc::ld16(t_s + c16 * 16, v);
          tc::wait_ld();
          #pragma unroll
          for (int i = 0; i < 16; ++i) x[c16 * 16 + i] = __uint_as_float(v[i]);
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);

        // scale, softcap, band + causal predicate, tile max
        float mx = -INFINITY;
        #pragma unroll
        for (int k = 0; k < BN; ++k) {
          const int key = key0 + k;
          float v = x[k];
          v = use_cap ? softcap_tanh(v * scale, softcap, inv_cap) * kLog2e : v * scale_l2;
          const bool vis = row_ok && key <= p && (window == 0 || p - key < window);
          v = vis ? v : -INFINITY;
          x[k] = v;
          mx = fmaxf(mx, v);
        }
        const float m_cand = fmaxf(m_run, mx);
        if (m_cand > m_run + kRescaleThreshold) {  // lazy rescale (also the first visible key)
          alpha = exp2f(m_run - m_cand);
          m_run = m_cand;
        }
      }
      // P_{j-1} has been multiplied in and O is stable once PV_{j-1} is done
      if (okw && j > 0) {
        okw = __all_sync(0xffffffffu, mbar_wait(&bars->pv_done, (j - 1) & 1));
        tc::fence_after();
        if (okw && __any_sync(0xffffffffu, alpha != 1.f)) {
          #pragma unroll 1
          for (int c16 = 0; c16 < C::kOCols / 16; ++c16) {
            uint32_t v[16];
            tc::ld16(t_o + c16 * 16, v);
            tc::wait_ld();
            #pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tc::st16(t_o + c16 * 16, v);
          }
          tc::wait_st();
        }
      }
      if (okw) {
        // zero V rows that no row of this tile can see (first / last key tile)
        if (j == 0 || j == nkt - 1) {
          uint8_t* st = stages + (j & 1) * C::kStageBytes;
          uint8_t* vt = KEQV ? st + dh * C::kVChunks * C::kChunkTileBytes : st + C::kKBytes;
          const int z_lo = max(0, j_lo - key0);       // rows [0, z_lo) hidden
          const int z_hi = min(BN, j_hi - key0 + 1);  // rows [z_hi, BN) hidden
          if (z_lo > 0 || z_hi < BN) {
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
        // P = exp2(x - m): bf16 high part and bf16 remainder into tensor memory
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        float psum = 0.f;
        #pragma unroll
        for (int c32 = 0; c32 < BN / 32; ++c32) {
          uint32_t hi[16], lo[16];
          #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = exp2f(x[c32 * 32 + 2 * i] - m_use);
            const float bb = exp2f(x[c32 * 32 + 2 * i + 1] - m_use);
            psum += a + bb;
            hi[i] = pack_bf16x2(a, bb);
            const float2 hf = unpack_bf16x2(hi[i]);
            lo[i] = pack_bf16x2(a - hf.x, bb - hf.y);
          }
          tc::st16(tmem + lane_off + C::kTmemPhi + c32 * 16, hi);
          tc::st16(tmem + lane_off + C::kTmemPlo + c32 * 16, lo);
        }
        l_run = l_run * alpha + psum;
        tc::wait_st();
        tc::fence_before();
      }
      if (!okw && lane == 0) {
        flag_error(err, PSW_DEVERR_PIPELINE);
        *sm_abort = 1;
      }
      named_bar_sync(1, kSoftmaxWarps * 32);  // V zeroing of all softmax threads done
      if (*sm_abort) break;
      if (lane == 0) mbar_arrive(&bars->p_full);
    }
    bool ok = !*sm_abort;

    // epilogue: O / l to global, lse
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->pv_done, (nkt - 1) & 1));
    tc::fence_after();
    if (ok) {
      const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
      float* orow = out + (static_cast<int64_t>(q0 + i0 + t) * n_q + kvh * group + h) * HD +
                    dh * C::kOCols;
      #pragma unroll 1
      for (int c16 = 0; c16 < C::kOCols / 16; ++c16) {
        uint32_t v[16];
        tc::ld16(t_o + c16 * 16, v);
        tc::wait_ld();
        if (row_ok) {
          #pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(orow + c16 * 16 + i) =
                make_float4(__uint_as_float(v[i]) * inv_l, __uint_as_float(v[i + 1]) * inv_l,
                            __uint_as_float(v[i + 2]) * inv_l, __uint_as_float(v[i + 3]) * inv_l);
        }
      }
      if (row_ok && dh == 0 && lse != nullptr)
        lse[static_cast<int64_t>(q0 + i0 + t) * n_q + kvh * group + h] =
            (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    } else if (lane == 0) {
      flag_error(err, PSW_DEVERR_PIPELINE);
      *abort_flag = 1;  // stops the producer and the MMA issuer
    }
  }

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
