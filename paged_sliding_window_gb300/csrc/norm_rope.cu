// norm_rope.cu -- the step before attention, fused: per-head RMS-norm of the
// new tokens' q, k and v, the proportional rotary embedding of q and k, and
// the cache write of k and v into their pages.
//
// Method (what is computed), per head vector x of head_dim elements at
// absolute position pos (token t of sequence b: pos = past_b + t - cu_new[b]):
//   y_d = x_d / sqrt(mean(x^2) + eps) * w_d
// (RMS-norm of each head vector before the rotation: InfiniLM PR 581 "feat:
// support gemma2 and gemma3_text", Gemma-3 item 1, whose weights are loaded
// as 1 + the stored value; v is normalised too: "MNN supports the full Gemma4
// family", section 6.1), then for q and k only (V is not rotated: same page,
// section 6.2) the proportional rotary embedding of "Gemma 4 model
// architecture analysis", challenge 5: pair i of dims (i, i + head_dim/2)
// turns by pos * theta^(-2i/head_dim) for i < rope_angles and not at all
// beyond (the zero-padded frequencies), theta 1e4 on sliding layers and 1e6
// on full ones. The normalised K and V rows go straight into their slots,
// block_table[b][pos / 16] * 16 + pos % 16 (section 6.3 of that page).
//
// Design (how, on sm_103a): the kernel is HBM-bound on a prefill-sized step
// and latency-bound on a decode step, and what costs time is the chain of
// dependent steps per token (find the sequence, read its past length and
// block id, form the angles), not arithmetic. A CTA (8 warps, 16 at
// head_dim 512; about one wave of them) owns tokens t, t + grid, ... It
// resolves up to 256 of them at once, thread j taking the j-th (sequence by
// binary search over the offsets staged in shared memory, position, slot),
// then runs them as a two-stage pipeline: while token j is computed, the
// rows of token j + 1 are in flight (each warp loads up to four head
// vectors, 16 or 32 bytes per lane each); its angles are formed at the
// barrier between the two. An angle is pos * freq reduced to [-pi, pi] in
// double, from frequencies the host computed in double (a float product
// would lose about 0.006 rad at position 65536, far more than a bf16 unit),
// with its sine and cosine in float. Computing a head vector: the sum of
// squares reduced with shuffles, the norm's scale and weight, the rotation
// of q and k (the partner of lane l's elements is held by lane l ^ 16: lanes
// 0-15 hold the first half of the head, 16-31 the second), one rounding to
// bf16, 16-byte stores to q_out or into the token's page slot.
#include <math.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace {

constexpr int kNrStaged = 1024;  // cu_new entries staged in shared memory
constexpr int kNrChunk = 256;    // tokens of a CTA resolved together
constexpr double kTwoPiHi = 6.283185307179586;       // 2 pi rounded to double
constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi - kTwoPiHi

// theta^(-2i / head_dim) for the rotated pairs, 0 beyond: computed on the host
// in double and passed by value, so no CTA spends double-precision
// exponentials on it.
struct FreqTable {
  double f[256];
  float2 f2[256];  // the same split into a float and the float of the rest
};

// 2 pi in three floats (each the float nearest to what the previous ones
// leave) and 1 / (2 pi) rounded to float, for the angle reduction below.
constexpr float kC1 = 6.2831854820251465f;
constexpr float kC2 = -1.7484555314695172e-7f;
constexpr float kC3 = -6.8604980400235275e-15f;
constexpr float kInvTwoPi = 0.15915493667125702f;

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Per-token state of one pipeline stage: the token, its position and slot,
// its rotation (cos, sin) per pair.
template <int HD>
struct TokenStage {
  // (cos, -sin) for the first half of the head, (cos, sin) for the second:
  // out = y cos + partner * (signed sin) on either side
  float2 cs[2][HD / 2];
  long long slot;  // K/V slot, -1: no cache write
  int pos;         // -1: token skipped
};

template <int HD, int WARPS, int ITEMS>
struct NormRope {
  static constexpr int kThreads = WARPS * 32;
  static constexpr int kHalf = HD / 2;
  static constexpr int kPer = HD / 32;    // elements per lane
  static constexpr int kVecs = kPer / 8;  // 16-byte accesses per lane per vector
};

template <int HD, int WARPS, int ITEMS>
__global__ void __launch_bounds__(WARPS * 32)
qkv_norm_rope_kernel(const __grid_constant__ FreqTable freq, const __nv_bfloat16* q,
                     const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                     const int32_t* __restrict__ cu_new, const int32_t* __restrict__ past_lens,
                     int n_seqs, const int32_t* __restrict__ block_table, int max_blocks,
                     int64_t num_blocks, int n_q, int n_kv, float eps,
                     const float* __restrict__ qw, const float* __restrict__ kw,
                     const float* __restrict__ vw, int rope_angles,
                     __nv_bfloat16* q_out,  // may be q itself: each lane rewrites what it read
                     __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool,
                     int32_t* err) {
  using C = NormRope<HD, WARPS, ITEMS>;
  constexpr int kPer = C::kPer, kVecs = C::kVecs, kHalf = C::kHalf;
  __shared__ int32_t s_cu[kNrStaged];
  __shared__ TokenStage<HD> s_st[2];
  __shared__ long long s_slots[kNrChunk];  // the CTA's next kNrChunk tokens: slot
  __shared__ int s_poss[kNrChunk];         // and position (-1: skipped)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool staged = n_seqs < kNrStaged;  // uniform over the grid
  if (staged)
    for (int i = tid; i <= n_seqs; i += C::kThreads) s_cu[i] = cu_new[i];
  __syncthreads();
  auto cu = [&](int i) { return staged ? s_cu[i] : cu_new[i]; };
  const int total = cu(n_seqs);
  const bool has_k = k != nullptr, has_v = v != nullptr;
  const int nvec = n_q + (has_k ? n_kv : 0) + (has_v ? n_kv : 0);

  // loads of token t's head vectors warp, warp + WARPS, ... into r
  auto load_rows = [&](int t, uint4 (&r)[ITEMS][kVecs]) {
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const int w = warp + u * WARPS;
      if (w >= nvec) continue;  // uniform over the warp
      const __nv_bfloat16* src;
      if (w < n_q)
        src = q + (static_cast<int64_t>(t) * n_q + w) * HD;
      else if (has_k && w < n_q + n_kv)
        src = k + (static_cast<int64_t>(t) * n_kv + (w - n_q)) * HD;
      else
        src = v + (static_cast<int64_t>(t) * n_kv + (w - n_q - (has_k ? n_kv : 0))) * HD;
      const uint4* s4 = reinterpret_cast<const uint4*>(src) + lane * kVecs;
#pragma unroll
      for (int c = 0; c < kVecs; ++c) r[u][c] = s4[c];
    }
  };
  // sequence, position and slot of token t
  auto resolve = [&](int t, int& pos_out, long long& slot_out) {
    int lo = 0, hi = n_seqs;  // sequence owning token t: largest b with cu_new[b] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu(mid) <= t) lo = mid; else hi = mid;
    }
    const int b = lo, start = cu(b);
    int pos = -1;
    long long slot = -1;
    if (t < start || t >= cu(b + 1)) {
      flag_error(err, PSW_DEVERR_LENGTH);  // offsets not monotone
    } else {
      const long long p = static_cast<long long>(past_lens[b]) + (t - start);
      if (p < 0 || p > 0x7fffffffLL) {
        flag_error(err, PSW_DEVERR_LENGTH);
      } else {
        pos = static_cast<int>(p);
        if (has_k) {
          const long long page = p / kBlockSize;
          if (page >= max_blocks) {
            flag_error(err, PSW_DEVERR_CAPACITY);
          } else {
            const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + page];
            if (blk < 0 || blk >= num_blocks)
              flag_error(err, PSW_DEVERR_BLOCK_ID);
            else
              slot = static_cast<long long>(blk) * kBlockSize + p % kBlockSize;
          }
        }
      }
    }
    pos_out = pos;
    slot_out = slot;
  };
  // all threads: the rotation of stage st's token at position pos
  auto angles = [&](TokenStage<HD>& st, int pos) {
    for (int i = tid; i < kHalf; i += C::kThreads) {
      float c = 1.f, sn = 0.f;
      if (pos >= 0 && i < rope_angles) {
        float r;
        if (pos < (1 << 24)) {
          // pos f = ph + pl from the float parts of f (pos is exact in a
          // float, ph's rounding error comes back exactly from the FMA), then
          // Cody-Waite reduction by the three-float 2 pi: each FMA multiplies
          // exactly and rounds once, so |r - (pos f mod 2 pi)| stays below
          // about 4e-7 for f <= 1
          const float pf = static_cast<float>(pos);
          const float2 fq = freq.f2[i];
          const float ph = pf * fq.x;
          const float pl = fmaf(pf, fq.y, fmaf(pf, fq.x, -ph));
          const float n = rintf(ph * kInvTwoPi);
          r = fmaf(-n, kC3, fmaf(-n, kC2, fmaf(-n, kC1, ph))) + pl;
        } else {  // beyond 2^24 the product needs double
          const double a = static_cast<double>(pos) * freq.f[i];
          const double n = rint(a * (1.0 / kTwoPiHi));
          r = static_cast<float>(fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, a)));  // |r| <= pi
        }
        sincosf(r, &sn, &c);
      }
      st.cs[0][i] = make_float2(c, -sn);
      st.cs[1][i] = make_float2(c, sn);
    }
  };
  // every warp: normalise, rotate and store its vectors of token t
  auto compute = [&](int t, const uint4 (&r)[ITEMS][kVecs], const TokenStage<HD>& st) {
    if (st.pos < 0) return;
    const long long slot = st.slot;
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const int w = warp + u * WARPS;
      if (w >= nvec) continue;  // uniform over the warp
      __nv_bfloat16* dst;
      const float* wt;
      bool rot;
      if (w < n_q) {
        dst = q_out + (static_cast<int64_t>(t) * n_q + w) * HD;
        wt = qw;
        rot = true;
      } else if (has_k && w < n_q + n_kv) {
        dst = slot >= 0 ? k_pool + (slot * n_kv + (w - n_q)) * HD : nullptr;
        wt = kw;
        rot = true;
      } else {
        dst = slot >= 0 ? v_pool + (slot * n_kv + (w - n_q - (has_k ? n_kv : 0))) * HD
                        : nullptr;
        wt = vw;
        rot = false;
      }
      if (dst == nullptr) continue;
      float y[kPer];
#pragma unroll
      for (int c = 0; c < kVecs; ++c) {
        const uint32_t wd[4] = {r[u][c].x, r[u][c].y, r[u][c].z, r[u][c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[c * 8 + 2 * e] = __uint_as_float(wd[e] << 16);
          y[c * 8 + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
        }
      }
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      // MUFU reciprocal square root: about 2^-22 relative, far inside the
      // error allowed before the bf16 rounding
      const float inv = rsqrtf(ss * (1.f / HD) + eps);
      if (wt != nullptr) {
        const float4* w4 = reinterpret_cast<const float4*>(wt) + lane * (kPer / 4);
#pragma unroll
        for (int c = 0; c < kPer / 4; ++c) {
          const float4 ww = __ldg(w4 + c);
          y[4 * c] *= inv * ww.x;
          y[4 * c + 1] *= inv * ww.y;
          y[4 * c + 2] *= inv * ww.z;
          y[4 * c + 3] *= inv * ww.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) y[e] *= inv;
      }
      if (rot) {
        const float4* cs4 =
            reinterpret_cast<const float4*>(st.cs[lane >> 4] + (lane & 15) * kPer);
#pragma unroll
        for (int e2 = 0; e2 < kPer / 2; ++e2) {  // two pairs per 16-byte read
          const float4 cc = cs4[e2];
          const float o0 = __shfl_xor_sync(0xffffffffu, y[2 * e2], 16);
          const float o1 = __shfl_xor_sync(0xffffffffu, y[2 * e2 + 1], 16);
          y[2 * e2] = fmaf(y[2 * e2], cc.x, o0 * cc.y);
          y[2 * e2 + 1] = fmaf(y[2 * e2 + 1], cc.z, o1 * cc.w);
        }
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst) + lane * kVecs;
#pragma unroll
      for (int c = 0; c < kVecs; ++c)
        d4[c] = make_uint4(pack_bf16_rn(y[c * 8], y[c * 8 + 1]),
                           pack_bf16_rn(y[c * 8 + 2], y[c * 8 + 3]),
                           pack_bf16_rn(y[c * 8 + 4], y[c * 8 + 5]),
                           pack_bf16_rn(y[c * 8 + 6], y[c * 8 + 7]));
    }
  };

  // This CTA's tokens are t = blockIdx.x + j * grid. Their positions and
  // slots are resolved kNrChunk at a time, thread j taking token j, so no
  // dependent lookup chain sits between two tokens. Tokens then run as a
  // two-stage pipeline: while token j is computed, the rows of token j + 1
  // are in flight; its angles are formed at the barrier between them. The
  // loop is unrolled by two so that both row buffers stay in registers.
  uint4 ra[ITEMS][kVecs], rb[ITEMS][kVecs];
  const int G = static_cast<int>(gridDim.x);
  const int n_mine = total > static_cast<int>(blockIdx.x)
                         ? (total - static_cast<int>(blockIdx.x) + G - 1) / G
                         : 0;
  for (int c0 = 0; c0 < n_mine; c0 += kNrChunk) {
    const int nc = min(kNrChunk, n_mine - c0);
    auto tok = [&](int j) { return static_cast<int>(blockIdx.x) + (c0 + j) * G; };
    load_rows(tok(0), ra);  // independent of every lookup
    for (int j = tid; j < nc; j += C::kThreads) resolve(tok(j), s_poss[j], s_slots[j]);
    __syncthreads();
    s_st[0].pos = s_poss[0];
    s_st[0].slot = s_slots[0];
    angles(s_st[0], s_poss[0]);
    __syncthreads();
    for (int j = 0; j < nc;) {
      // ---- token j from ra / stage 0, token j + 1 prepared into rb / stage 1
      if (j + 1 < nc) load_rows(tok(j + 1), rb);
      compute(tok(j), ra, s_st[0]);
      if (++j >= nc) break;
      if (tid == 0) { s_st[1].pos = s_poss[j]; s_st[1].slot = s_slots[j]; }
      angles(s_st[1], s_poss[j]);
      __syncthreads();
      // ---- token j from rb / stage 1, token j + 1 prepared into ra / stage 0
      if (j + 1 < nc) load_rows(tok(j + 1), ra);
      compute(tok(j), rb, s_st[1]);
      if (++j >= nc) break;
      if (tid == 0) { s_st[0].pos = s_poss[j]; s_st[0].slot = s_slots[j]; }
      angles(s_st[0], s_poss[j]);
      __syncthreads();
    }
    __syncthreads();  // the chunk arrays are rewritten by the next chunk
  }
}

template <int HD, int WARPS>
cudaError_t launch_items(int items, const FreqTable& ft, int grid, cudaStream_t stream,
                         const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                         const int32_t* cu_new, const int32_t* past_lens, int n_seqs,
                         const int32_t* block_table, int max_blocks, int64_t num_blocks, int n_q,
                         int n_kv, float eps, const float* qw, const float* kw, const float* vw,
                         int rope_angles, __nv_bfloat16* qo, __nv_bfloat16* kp,
                         __nv_bfloat16* vp, int32_t* err) {
#define PSW_NR_LAUNCH(I)                                                                      \
  qkv_norm_rope_kernel<HD, WARPS, I><<<grid, WARPS * 32, 0, stream>>>(                        \
      ft, q, k, v, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, n_q, n_kv, \
      eps, qw, kw, vw, rope_angles, qo, kp, vp, err)
  if (items <= 1) PSW_NR_LAUNCH(1);
  else if (items <= 2) PSW_NR_LAUNCH(2);
  else if (items <= 3) PSW_NR_LAUNCH(3);
  else PSW_NR_LAUNCH(4);
#undef PSW_NR_LAUNCH
  return cudaGetLastError();
}

}  // namespace

int launch_qkv_norm_rope(const LayerArgs& L, const NormRopeArgs& R, const void* q, const void* k,
                         const void* v, const int32_t* cu_new, const int32_t* past_lens,
                         int n_seqs, const int32_t* block_table, int max_blocks,
                         int64_t num_blocks, void* q_out, void* k_pool, void* v_pool, int num_sms,
                         int32_t* err, cudaStream_t stream) {
  FreqTable ft;
  const double log_theta = log(static_cast<double>(R.theta));
  for (int i = 0; i < 256; ++i) {
    ft.f[i] = (i < L.hd / 2 && i < R.rope_angles)
                  ? exp(-2.0 * static_cast<double>(i) / L.hd * log_theta)
                  : 0.0;
    const float hi = static_cast<float>(ft.f[i]);
    ft.f2[i] = make_float2(hi, static_cast<float>(ft.f[i] - static_cast<double>(hi)));
  }
  const int nvec = L.n_q + (k != nullptr ? L.n_kv : 0) + (v != nullptr ? L.n_kv : 0);
  // 8 warps (16 at head_dim 512), each holding up to 4 head vectors of a
  // token per stage
  const int warps = L.hd == 256 ? 8 : 16;
  const int items = (nvec + warps - 1) / warps;
  if (items > 4) return PSW_EINVAL_HEADS;
  const int grid = num_sms * (L.hd == 256 ? 3 : 2);  // about one wave of resident CTAs
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* qo = static_cast<__nv_bfloat16*>(q_out);
  auto* kp = static_cast<__nv_bfloat16*>(k_pool);
  auto* vp = static_cast<__nv_bfloat16*>(v_pool);
  const cudaError_t e =
      L.hd == 256
          ? launch_items<256, 8>(items, ft, grid, stream, qb, kb, vb, cu_new, past_lens, n_seqs,
                                 block_table, max_blocks, num_blocks, L.n_q, L.n_kv, R.eps,
                                 R.q_weight, R.k_weight, R.v_weight, R.rope_angles, qo, kp, vp,
                                 err)
          : launch_items<512, 16>(items, ft, grid, stream, qb, kb, vb, cu_new, past_lens, n_seqs,
                                  block_table, max_blocks, num_blocks, L.n_q, L.n_kv, R.eps,
                                  R.q_weight, R.k_weight, R.v_weight, R.rope_angles, qo, kp, vp,
                                  err);
  return e == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace psw

