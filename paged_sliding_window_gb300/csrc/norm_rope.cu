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
// Design (how, on sm_103a): the step is HBM-bound on a prefill-sized batch
// and latency-bound on a decode batch; no block-wide barrier sits on its
// path. A unit is NH head vectors of one tensor of one token (NH = 4, 2 or 1
// at head_dim 256, the largest dividing both head counts; 1 at head_dim
// 512), so every unit is full and one code path serves them all. Each warp
// of a persistent grid (as many CTAs as fit on the SMs) takes a contiguous
// block of units in token order, so consecutive units mostly share a token
// whose position, page slot and rotation it keeps. Two register buffers
// hold rows: the next unit's loads are in flight while one is processed.
// The sequence of a token is found by the whole warp, which splits the
// offsets 31 ways per round of coalesced loads (one round up to 31
// sequences, two up to 961), reading past_lens in the last round. Lane l
// holds elements [l m, l m + m) of each half of a head vector (m =
// head_dim / 64), so the two elements of every rotation pair sit in the
// same lane: the lane forms the rotation of its m pairs once per token and
// rotates without shuffles. An angle is pos * freq reduced to [-pi/4, pi/4]
// and a quadrant: below position 2^24 in float, from the two-float split of
// a frequency the host computed in double, by Cody-Waite with a three-float
// pi / 2 (plus a second step for the rounding of the quadrant above 2^22),
// in double beyond; its sine and cosine from Taylor polynomials and the
// quadrant's symmetry, 2.2e-7 at most in all. The sums of squares of a
// unit's rows are reduced together (one halving shuffle tree, one
// reciprocal square root per lane); the norm's weight and the rotation are
// folded into per-element coefficients; one rounding to bf16; 8- or
// 16-byte stores to q_out or into the token's page slot.
#include <math.h>

#include <atomic>
#include <type_traits>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace {

constexpr int kThreads = 256;  // 8 warps per CTA, each on its own units

// theta^(-2i / head_dim) for the rotated pairs, 0 beyond: computed on the host
// in double and passed by value, so no CTA spends double-precision
// exponentials on it.
struct FreqTable {
  double f[256];
  float2 f2[256];  // the same split into a float and the float of the rest
};

// pi / 2 in three floats (each the float nearest to what the previous ones
// leave; a quarter of the same split of 2 pi, exact in binary) and 2 / pi
// rounded to float, for the angle reduction below.
constexpr float kP1 = 1.5707963705062866f;
constexpr float kP2 = -4.3711388286737929e-8f;
constexpr float kP3 = -1.7151245100058819e-15f;
constexpr float kTwoOverPi = 0.63661974668502808f;
constexpr double kHalfPiHi = 1.5707963267948966;      // pi / 2 rounded to double
constexpr double kHalfPiLo = 6.123233995736766e-17;   // pi / 2 - kHalfPiHi

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// sin and cos of x + qd pi / 2 for |x| <= pi / 4 (a little beyond after
// rounding): the Taylor series of sin through x^9 and of cos through x^8
// (truncation below 1.8e-9 and 2.5e-8 at pi / 4), then the quadrant's
// symmetry: (sin, cos) of x + pi / 2 is (cos x, -sin x), of x + pi is
// (-sin x, -cos x), of x + 3 pi / 2 is (-cos x, sin x).
__device__ __forceinline__ void sincos_quadrant(float x, int qd, float& sn, float& cs) {
  const float x2 = x * x;
  float sp = fmaf(x2, 1.f / 362880.f, -1.f / 5040.f);
  sp = fmaf(x2, sp, 1.f / 120.f);
  sp = fmaf(x2, sp, -1.f / 6.f);
  const float sx = fmaf(x * x2, sp, x);
  float cp = fmaf(x2, 1.f / 40320.f, -1.f / 720.f);
  cp = fmaf(x2, cp, 1.f / 24.f);
  cp = fmaf(x2, cp, -0.5f);
  const float cx = fmaf(x2, cp, 1.f);
  const float s0 = (qd & 1) ? cx : sx;
  const float c0 = (qd & 1) ? sx : cx;
  sn = __uint_as_float(__float_as_uint(s0) ^ ((qd & 2) ? 0x80000000u : 0u));
  cs = __uint_as_float(__float_as_uint(c0) ^ (((qd + 1) & 2) ? 0x80000000u : 0u));
}

// bf16 -> float of the low and high half of a word by byte permutes, as
// volatile asm: the rows are unpacked once for the sums of squares and again
// for the results, and the second unpack must not be merged with the first
// (that would keep every unpacked row live across the reduction).
__device__ __forceinline__ float2 unpack_again(uint32_t w) {
  uint32_t lo, hi;
  asm volatile("prmt.b32 %0, %2, 0, 0x1044;\n\tprmt.b32 %1, %2, 0, 0x3244;"
               : "=r"(lo), "=r"(hi)
               : "r"(w));
  return make_float2(__uint_as_float(lo), __uint_as_float(hi));
}

// A lane's share of one half of a head vector: HD / 64 bf16 values, one
// 8-byte (head_dim 256) or 16-byte (head_dim 512) access.
template <int HD>
struct Share;
template <>
struct Share<256> {
  using T = uint2;
  __device__ static void unpack(const T& r, float (&y)[4]) {
    y[0] = __uint_as_float(r.x << 16);
    y[1] = __uint_as_float(r.x & 0xFFFF0000u);
    y[2] = __uint_as_float(r.y << 16);
    y[3] = __uint_as_float(r.y & 0xFFFF0000u);
  }
  __device__ static void unpack_again(const T& r, float (&y)[4]) {
    const float2 a = psw::unpack_again(r.x), b = psw::unpack_again(r.y);
    y[0] = a.x, y[1] = a.y, y[2] = b.x, y[3] = b.y;
  }
  __device__ static T pack(const float (&y)[4]) {
    return make_uint2(pack_bf16_rn(y[0], y[1]), pack_bf16_rn(y[2], y[3]));
  }
};
template <>
struct Share<512> {
  using T = uint4;
  __device__ static void unpack(const T& r, float (&y)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y[2 * e] = __uint_as_float(w[e] << 16);
      y[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  __device__ static void unpack_again(const T& r, float (&y)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = psw::unpack_again(w[e]);
      y[2 * e] = a.x, y[2 * e + 1] = a.y;
    }
  }
  __device__ static T pack(const float (&y)[8]) {
    return make_uint4(pack_bf16_rn(y[0], y[1]), pack_bf16_rn(y[2], y[3]),
                      pack_bf16_rn(y[4], y[5]), pack_bf16_rn(y[6], y[7]));
  }
};

// Warp sums of VB values at once (x[j]: this lane's part of sum j). Each
// round halves the list: a lane keeps one half, sends the other to its
// partner across lane bit 16, 8, ... and adds what it receives; after
// log2(VB) rounds lane l holds a partial of sum l / (32 / VB), which the
// remaining xor rounds complete. VB - 1 + 5 - log2(VB) shuffles in all.
template <int VB>
__device__ __forceinline__ float warp_sums(float (&x)[VB], int lane) {
#pragma unroll
  for (int r = 0; (VB >> r) > 1; ++r) {
    const int n = VB >> r, mask = 16 >> r;
    const bool up = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? x[i + n / 2] : x[i];
      const float send = up ? x[i] : x[i + n / 2];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
  }
  float m = x[0];
#pragma unroll
  for (int mask = 16 / VB; mask > 0; mask >>= 1) m += __shfl_xor_sync(0xffffffffu, m, mask);
  return m;  // the sum number lane / (32 / VB)
}

// The sequence of token t, found by the whole warp: b is the largest index
// below n_seqs with cu_new[b] <= t. Each round the lanes probe the open range
// at 31 evenly spaced offsets (one coalesced load), and the ballot of
// "offset <= t" narrows it to one stride; the last round (range of at most
// 31) probes every index plus the range's end, so it also yields
// cu_new[b + 1], and it reads past_lens alongside. False when t lies before
// cu_new[0] or outside [cu_new[b], cu_new[b + 1]) (offsets not monotone).
// Every lane returns the same values.
__device__ __forceinline__ bool find_sequence(const int32_t* __restrict__ cu_new,
                                              const int32_t* __restrict__ past_lens,
                                              int n_seqs, int t, int lane, int& b, int& start,
                                              int& end, int& past) {
  int lo = 0, hi = n_seqs;  // b in [lo, hi)
  while (hi > lo) {
    const int step = (hi - lo + 30) / 31;
    const int idx = lo + lane * step;
    const int c = idx <= hi ? __ldg(cu_new + idx) : 0;
    const int pl = (step == 1 && idx < hi) ? __ldg(past_lens + idx) : 0;
    const unsigned m = __ballot_sync(0xffffffffu, idx < hi && c <= t);
    if (m == 0) return false;
    const int h = 31 - __clz(static_cast<int>(m));
    if (step == 1) {  // h <= 30: lane h + 1 holds cu_new[b + 1]
      b = lo + h;
      start = __shfl_sync(0xffffffffu, c, h);
      end = __shfl_sync(0xffffffffu, c, h + 1);
      past = __shfl_sync(0xffffffffu, pl, h);
      return t < end;
    }
    lo += h * step;
    hi = min(hi, lo + step);
  }
  return false;
}

// NH head vectors of one tensor of one token form a unit; the host picks NH
// so that every unit is full (a power of two dividing n_q and n_kv).
template <int HD, int NH>
__global__ void __launch_bounds__(kThreads, 2)  // two CTAs per SM: 128 registers
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
  constexpr int kM = HD / 64;  // elements of each half per lane
  using S = Share<HD>;
  using Vec = typename S::T;
  // the split frequencies, [e][lane] so that a warp's reads are contiguous
  __shared__ float2 s_fq[kM][32];
  for (int i = threadIdx.x; i < HD / 2; i += kThreads) s_fq[i % kM][i / kM] = freq.f2[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const bool has_k = k != nullptr, has_v = v != nullptr;
  // units of a token: q heads, then k heads, then v heads, NH at a time
  const int uq = n_q / NH, uk = has_k ? n_kv / NH : 0, uv = has_v ? n_kv / NH : 0;
  const int n_u = uq + uk + uv;
  const int total = __ldg(cu_new + n_seqs);
  if (total <= 0) return;
  // this warp's units: a contiguous block, so that consecutive units mostly
  // share a token (its position, slot and rotation are kept)
  const int64_t n_units = static_cast<int64_t>(total) * n_u;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t per = (n_units + n_warps - 1) / n_warps;
  const int64_t u0 = warp_id * per;
  if (u0 >= n_units) return;
  const int count = static_cast<int>(min(per, n_units - u0));
  int t = static_cast<int>(u0 / n_u), g = static_cast<int>(u0 - (u0 / n_u) * n_u);

  // the sequence of the last token met: tokens [s_start, s_end)
  int s_b = 0, s_start = 1, s_end = 0, s_past = 0;
  int pos_t = -1, pos = 0;        // token whose position pos is known (-1: none)
  int slot_t = -1;                // token whose page slot is known
  int64_t slot = -1;
  int rot_t = -1;                 // token whose rotation is in (rc, rs)
  float rc[kM], rs[kM];

  auto row_ptr = [&](int tt, int gg) -> const __nv_bfloat16* {
    if (gg < uq) return q + (static_cast<int64_t>(tt) * n_q + gg * NH) * HD + lane * kM;
    if (gg < uq + uk) return k + (static_cast<int64_t>(tt) * n_kv + (gg - uq) * NH) * HD + lane * kM;
    return v + (static_cast<int64_t>(tt) * n_kv + (gg - uq - uk) * NH) * HD + lane * kM;
  };
  auto load = [&](int tt, int gg, Vec (&ra)[NH], Vec (&rb)[NH]) {
    const __nv_bfloat16* src = row_ptr(tt, gg);
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      ra[j] = *reinterpret_cast<const Vec*>(src + j * HD);
      rb[j] = *reinterpret_cast<const Vec*>(src + j * HD + HD / 2);
    }
  };
  // position of token tt; false: the token is skipped (flagged)
  auto position = [&](int tt) -> bool {
    if (tt == pos_t) return true;
    if (!(tt >= s_start && tt < s_end)) {
      if (!find_sequence(cu_new, past_lens, n_seqs, tt, lane, s_b, s_start, s_end, s_past)) {
        if (lane == 0) flag_error(err, PSW_DEVERR_LENGTH);
        s_start = 1;
        s_end = 0;
        return false;
      }
    }
    const int64_t p = static_cast<int64_t>(s_past) + (tt - s_start);
    if (s_past < 0 || p > 0x7fffffffLL) {
      if (lane == 0) flag_error(err, PSW_DEVERR_LENGTH);
      return false;
    }
    pos = static_cast<int>(p);
    pos_t = tt;
    return true;
  };
  // page slot of token tt (at position pos); false: no cache write (flagged)
  auto page_slot = [&](int tt) -> bool {
    if (tt != slot_t) {
      slot_t = tt;
      slot = -1;
      const int page = pos / kBlockSize;
      if (page >= max_blocks) {
        if (lane == 0) flag_error(err, PSW_DEVERR_CAPACITY);
      } else {
        const int32_t blk = __ldg(block_table + static_cast<int64_t>(s_b) * max_blocks + page);
        if (blk < 0 || blk >= num_blocks) {
          if (lane == 0) flag_error(err, PSW_DEVERR_BLOCK_ID);
        } else {
          slot = static_cast<int64_t>(blk) * kBlockSize + pos % kBlockSize;
        }
      }
    }
    return slot >= 0;
  };
  // rotation of this lane's pairs i = lane kM + e at position pos
  auto rotation = [&](int tt) {
    if (tt == rot_t) return;
    rot_t = tt;
#pragma unroll
    for (int e = 0; e < kM; ++e) {
      const int i = lane * kM + e;
      float sn = 0.f, cs = 1.f;
      if (i < rope_angles) {
        float x;
        int qd;
        if (pos < (1 << 24)) {
          // pos f = ph + pl from the float parts of f (pos is exact in a
          // float, ph's rounding error comes back exactly from the FMA),
          // then Cody-Waite reduction by the three-float pi / 2: each FMA
          // multiplies exactly and rounds once
          const float2 fq = s_fq[e][lane];
          const float pf = static_cast<float>(pos);
          const float ph = pf * fq.x;
          const float pl = fmaf(pf, fq.y, fmaf(pf, fq.x, -ph));
          const float n1 = rintf(ph * kTwoOverPi);
          x = fmaf(-n1, kP3, fmaf(-n1, kP2, fmaf(-n1, kP1, ph))) + pl;
          // above 2^22 the float products behind n1 (ph, ph 2/pi) can put
          // it one or two off; x is still accurate for that n1, and a second
          // reduction of x (a few pi / 2 at most, exact products) brings it
          // back to [-pi/4, pi/4]
          const float n2 = rintf(x * kTwoOverPi);
          x = fmaf(-n2, kP2, fmaf(-n2, kP1, x));
          qd = static_cast<int>(n1) + static_cast<int>(n2);
        } else {  // beyond 2^24 the product needs double
          const double a = static_cast<double>(pos) * freq.f[i];
          const double n1 = rint(a * (1.0 / kHalfPiHi));
          x = static_cast<float>(fma(-n1, kHalfPiLo, fma(-n1, kHalfPiHi, a)));
          qd = static_cast<int>(static_cast<int64_t>(n1) & 3);
        }
        sincos_quadrant(x, qd, sn, cs);
      }
      rc[e] = cs;
      rs[e] = sn;
    }
  };
  // normalise, rotate (q, k) and store the unit (tt, gg) held in (ra, rb)
  auto process = [&](int tt, int gg, const Vec (&ra)[NH], const Vec (&rb)[NH]) {
    if (!position(tt)) return;
    const int kind = gg < uq ? 0 : (gg < uq + uk ? 1 : 2);
    __nv_bfloat16* dst;
    if (kind == 0) {
      dst = q_out + (static_cast<int64_t>(tt) * n_q + gg * NH) * HD + lane * kM;
    } else {
      if (!page_slot(tt)) return;
      const int h0 = (gg - (kind == 1 ? uq : uq + uk)) * NH;
      dst = (kind == 1 ? k_pool : v_pool) + (slot * n_kv + h0) * HD + lane * kM;
    }
    const float* wt = kind == 0 ? qw : (kind == 1 ? kw : vw);
    // per element coefficients: with the weights wa, wb and this lane's
    // rotation (cos, sin) of pair lane kM + e,
    //   out_a = inv (y_a wa cos - y_b wb sin), out_b = inv (y_b wb cos + y_a wa sin)
    // and out = inv y w for v
    float ca[kM], sa[kM], cb[kM], sb[kM];
#pragma unroll
    for (int c4 = 0; c4 < kM / 4; ++c4) {
      float4 a4 = make_float4(1.f, 1.f, 1.f, 1.f), b4 = a4;
      if (wt != nullptr) {
        a4 = __ldg(reinterpret_cast<const float4*>(wt + lane * kM) + c4);
        b4 = __ldg(reinterpret_cast<const float4*>(wt + HD / 2 + lane * kM) + c4);
      }
      ca[4 * c4] = a4.x, ca[4 * c4 + 1] = a4.y, ca[4 * c4 + 2] = a4.z, ca[4 * c4 + 3] = a4.w;
      cb[4 * c4] = b4.x, cb[4 * c4 + 1] = b4.y, cb[4 * c4 + 2] = b4.z, cb[4 * c4 + 3] = b4.w;
    }
    const bool rot = kind < 2;
    if (rot) {
      rotation(tt);
#pragma unroll
      for (int e = 0; e < kM; ++e) {
        sa[e] = ca[e] * rs[e];
        ca[e] *= rc[e];
        sb[e] = cb[e] * rs[e];
        cb[e] *= rc[e];
      }
    }
    // the sums of squares of the unit's rows, reduced together
    float ss[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      float ya[kM], yb[kM];
      S::unpack(ra[j], ya);
      S::unpack(rb[j], yb);
      ss[j] = 0.f;
#pragma unroll
      for (int e = 0; e < kM; ++e) ss[j] = fmaf(yb[e], yb[e], fmaf(ya[e], ya[e], ss[j]));
    }
    // MUFU reciprocal square root: about 2^-22 relative, far inside the
    // error allowed before the bf16 rounding
    const float inv_mine = rsqrtf(warp_sums<NH>(ss, lane) * (1.f / HD) + eps);
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      const float inv = __shfl_sync(0xffffffffu, inv_mine, j * (32 / NH));
      float ya[kM], yb[kM], oa[kM], ob[kM];
      S::unpack_again(ra[j], ya);
      S::unpack_again(rb[j], yb);
      if (rot) {
#pragma unroll
        for (int e = 0; e < kM; ++e) {
          oa[e] = inv * fmaf(ya[e], ca[e], -(yb[e] * sb[e]));
          ob[e] = inv * fmaf(yb[e], cb[e], ya[e] * sa[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kM; ++e) {
          oa[e] = inv * (ya[e] * ca[e]);
          ob[e] = inv * (yb[e] * cb[e]);
        }
      }
      *reinterpret_cast<Vec*>(dst + j * HD) = S::pack(oa);
      *reinterpret_cast<Vec*>(dst + j * HD + HD / 2) = S::pack(ob);
    }
  };
  auto next = [&](int& tt, int& gg) {
    if (++gg == n_u) {
      gg = 0;
      ++tt;
    }
  };

  // two register buffers: the next unit's rows are in flight while one is
  // processed
  Vec a0[NH], b0[NH], a1[NH], b1[NH];
  load(t, g, a0, b0);
  for (int c = 0; c < count; c += 2) {
    int t1 = t, g1 = g;
    next(t1, g1);
    if (c + 1 < count) load(t1, g1, a1, b1);
    process(t, g, a0, b0);
    if (c + 1 >= count) break;
    int t2 = t1, g2 = g1;
    next(t2, g2);
    if (c + 2 < count) load(t2, g2, a0, b0);
    process(t1, g1, a1, b1);
    t = t2;
    g = g2;
  }
}

// CTAs resident on an SM (registers decide it), asked once: the grid is
// that many per SM, so every CTA is resident from the start.
template <int HD, int NH>
int resident_ctas() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, qkv_norm_rope_kernel<HD, NH>, kThreads,
                                                      0) != cudaSuccess ||
        n < 1)
      n = 1;
    cached.store(n, std::memory_order_relaxed);
  }
  return n;
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
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* qo = static_cast<__nv_bfloat16*>(q_out);
  auto* kp = static_cast<__nv_bfloat16*>(k_pool);
  auto* vp = static_cast<__nv_bfloat16*>(v_pool);
  // head vectors per unit: the largest of 4, 2, 1 dividing the head counts
  // at head_dim 256, 1 at 512 (two units of rows per warp stay within its
  // registers)
  const bool kv = k != nullptr || v != nullptr;
  int nh = L.hd == 256 ? 4 : 1;
  while (nh > 1 && (L.n_q % nh != 0 || (kv && L.n_kv % nh != 0))) nh >>= 1;
#define PSW_NR_LAUNCH(HD_, NH_)                                                             \
  qkv_norm_rope_kernel<HD_, NH_><<<num_sms * resident_ctas<HD_, NH_>(), kThreads, 0, stream>>>( \
      ft, qb, kb, vb, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, L.n_q,  \
      L.n_kv, R.eps, R.q_weight, R.k_weight, R.v_weight, R.rope_angles, qo, kp, vp, err)
  if (L.hd == 256) {
    if (nh == 4) PSW_NR_LAUNCH(256, 4);
    else if (nh == 2) PSW_NR_LAUNCH(256, 2);
    else PSW_NR_LAUNCH(256, 1);
  } else {
    PSW_NR_LAUNCH(512, 1);
  }
#undef PSW_NR_LAUNCH
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

}  // namespace psw

