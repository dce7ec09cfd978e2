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
// Design (how, on sm_103a): the kernel is memory-bound and small (a decode
// step moves a few hundred KB), so it aims at few dependent round trips: one
// CTA per token (grid-stride), the token offsets staged in shared memory,
// the token's angles computed once per CTA and shared by all its heads, one
// warp per head vector with 16- or 32-byte loads per lane, the sum of squares
// reduced with shuffles, and the rotation partner of lane l's elements held
// by lane l ^ 16 (lanes 0-15 hold the first half of the head, 16-31 the
// second). The angle pos * freq is formed and reduced to [-pi, pi] in double
// (a float product would lose about 0.006 rad at position 65536, far more
// than a bf16 unit), then its sine and cosine are taken in float.
#include <math.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace {

constexpr int kNrThreads = 256;
constexpr int kNrWarps = kNrThreads / 32;
constexpr int kNrStaged = 2048;  // cu_new entries staged in shared memory
constexpr double kTwoPiHi = 6.283185307179586;       // 2 pi rounded to double
constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi - kTwoPiHi

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
__global__ void __launch_bounds__(kNrThreads)
qkv_norm_rope_kernel(const __nv_bfloat16* q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ cu_new,
                     const int32_t* __restrict__ past_lens, int n_seqs,
                     const int32_t* __restrict__ block_table, int max_blocks, int64_t num_blocks,
                     int n_q, int n_kv, float eps, const float* __restrict__ qw,
                     const float* __restrict__ kw, const float* __restrict__ vw,
                     double log_theta, int rope_angles,
                     __nv_bfloat16* q_out,  // may be q itself: each lane rewrites what it read
                     __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ v_pool,
                     int32_t* err) {
  constexpr int kHalf = HD / 2;
  constexpr int kPer = HD / 32;  // elements per lane
  constexpr int kVecs = kPer / 8;  // 16-byte vectors per lane
  __shared__ int32_t s_cu[kNrStaged];
  __shared__ double s_freq[kHalf];
  __shared__ float2 s_cs[kHalf];
  __shared__ long long s_slot;  // slot of the token's K/V row, -1: no cache write
  __shared__ int s_pos;         // position, -1: the token is skipped
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool staged = n_seqs < kNrStaged;  // uniform over the grid
  if (staged)
    for (int i = tid; i <= n_seqs; i += kNrThreads) s_cu[i] = cu_new[i];
  for (int i = tid; i < kHalf; i += kNrThreads)
    s_freq[i] = i < rope_angles ? exp(-2.0 * static_cast<double>(i) / HD * log_theta) : 0.0;
  __syncthreads();
  auto cu = [&](int i) { return staged ? s_cu[i] : cu_new[i]; };
  const int total = cu(n_seqs);
  const bool has_k = k != nullptr, has_v = v != nullptr;
  const int nvec = n_q + (has_k ? n_kv : 0) + (has_v ? n_kv : 0);

  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    if (tid == 0) {
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
      s_pos = pos;
      s_slot = slot;
    }
    __syncthreads();
    const int pos = s_pos;
    const long long slot = s_slot;
    if (pos >= 0) {
      for (int i = tid; i < kHalf; i += kNrThreads) {
        float c = 1.f, s = 0.f;
        if (i < rope_angles) {
          const double a = static_cast<double>(pos) * s_freq[i];
          const double n = rint(a * (1.0 / kTwoPiHi));
          const double r = fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, a));  // |r| <= pi
          sincosf(static_cast<float>(r), &s, &c);
        }
        s_cs[i] = make_float2(c, s);
      }
    }
    __syncthreads();
    if (pos >= 0) {
      for (int w = warp; w < nvec; w += kNrWarps) {
        const __nv_bfloat16* src;
        __nv_bfloat16* dst;
        const float* wt;
        bool rot;
        if (w < n_q) {
          src = q + (static_cast<int64_t>(t) * n_q + w) * HD;
          dst = q_out + (static_cast<int64_t>(t) * n_q + w) * HD;
          wt = qw;
          rot = true;
        } else if (has_k && w < n_q + n_kv) {
          const int g = w - n_q;
          src = k + (static_cast<int64_t>(t) * n_kv + g) * HD;
          dst = slot >= 0 ? k_pool + (slot * n_kv + g) * HD : nullptr;
          wt = kw;
          rot = true;
        } else {
          const int g = w - n_q - (has_k ? n_kv : 0);
          src = v + (static_cast<int64_t>(t) * n_kv + g) * HD;
          dst = slot >= 0 ? v_pool + (slot * n_kv + g) * HD : nullptr;
          wt = vw;
          rot = false;
        }
        if (dst == nullptr) continue;  // uniform over the warp
        float y[kPer];
        {
          const uint4* s4 = reinterpret_cast<const uint4*>(src) + lane * kVecs;
#pragma unroll
          for (int c = 0; c < kVecs; ++c) {
            const uint4 u = s4[c];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              y[c * 8 + 2 * e] = __uint_as_float(wd[e] << 16);
              y[c * 8 + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
            }
          }
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < kPer; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.f / sqrtf(ss / static_cast<float>(HD) + eps);
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
          const bool first_half = lane < 16;
#pragma unroll
          for (int e = 0; e < kPer; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, y[e], 16);
            const int i = (lane & 15) * kPer + e;  // pair index
            const float2 cs = s_cs[i];
            y[e] = first_half ? fmaf(y[e], cs.x, -other * cs.y) : fmaf(y[e], cs.x, other * cs.y);
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
    }
    __syncthreads();  // s_pos, s_slot and s_cs are rewritten for the next token
  }
}

}  // namespace

int launch_qkv_norm_rope(const LayerArgs& L, const NormRopeArgs& R, const void* q, const void* k,
                         const void* v, const int32_t* cu_new, const int32_t* past_lens,
                         int n_seqs, const int32_t* block_table, int max_blocks,
                         int64_t num_blocks, void* q_out, void* k_pool, void* v_pool, int num_sms,
                         int32_t* err, cudaStream_t stream) {
  const int grid = num_sms * 8;
  const double log_theta = log(static_cast<double>(R.theta));
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* qo = static_cast<__nv_bfloat16*>(q_out);
  auto* kp = static_cast<__nv_bfloat16*>(k_pool);
  auto* vp = static_cast<__nv_bfloat16*>(v_pool);
  if (L.hd == 256)
    qkv_norm_rope_kernel<256><<<grid, kNrThreads, 0, stream>>>(
        qb, kb, vb, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, L.n_q, L.n_kv,
        R.eps, R.q_weight, R.k_weight, R.v_weight, log_theta, R.rope_angles, qo, kp, vp, err);
  else
    qkv_norm_rope_kernel<512><<<grid, kNrThreads, 0, stream>>>(
        qb, kb, vb, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, L.n_q, L.n_kv,
        R.eps, R.q_weight, R.k_weight, R.v_weight, log_theta, R.rope_angles, qo, kp, vp, err);
  return cudaGetLastError() == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace psw
