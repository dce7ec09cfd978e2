// kv_cache_write.cu -- reshape_and_cache for 16-token pages.
//
// "Gemma 4 model architecture analysis" (vLLM-Kunlun), section 6.4: every new
// token's K and V rows are copied into key_cache[block_id, offset, :, :] of a
// [num_blocks][16][n_kv][head_dim] pool; the slot comes from the block table
// (section 6.3: block_table[b][pos / 16] * 16 + pos % 16), computed here from
// the table and the sequence's past length instead of a host-built
// slot_mapping array.
//
// One warp copies one token's row (n_kv * head_dim bf16, a multiple of 512 B)
// with 16-byte loads and stores; a grid-stride loop covers all tokens, whose
// count is read on the device (cu_new[n_seqs]).
#include <cuda_fp8.h>

#include "psw_internal.h"
#include "ptx.cuh"

namespace psw {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kStagedOffsets = 2048;  // cu_new entries staged in shared memory
constexpr int kPreVecs = 8;           // 16-byte vectors per lane loaded before the lookup

// The kernel is latency-bound (a few rows per block): the token offsets are
// staged in shared memory with one coalesced load, so the sequence search
// costs no global round trips, and each warp loads its token's new rows
// while it looks up the slot (past length, then block table).
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
kv_cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                      const int32_t* __restrict__ cu_new, const int32_t* __restrict__ past_lens,
                      int n_seqs, const int32_t* __restrict__ block_table, int max_blocks,
                      int64_t num_blocks, int row_vecs, uint4* __restrict__ k_pool,
                      uint4* __restrict__ v_pool, int32_t* err) {
  __shared__ int32_t s_cu[kStagedOffsets];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool staged = n_seqs < kStagedOffsets;  // uniform over the grid
  if (staged) {
    for (int i = threadIdx.x; i <= n_seqs; i += blockDim.x) s_cu[i] = cu_new[i];
    __syncthreads();
  }
  auto cu = [&](int i) { return staged ? s_cu[i] : cu_new[i]; };
  const int total = cu(n_seqs);
  const bool has_v = v_pool != nullptr;
  for (int t = blockIdx.x * kWarpsPerBlock + warp; t < total;
       t += gridDim.x * kWarpsPerBlock) {
    const uint4* ks = k + static_cast<int64_t>(t) * row_vecs;
    const uint4* vs = has_v ? v + static_cast<int64_t>(t) * row_vecs : nullptr;
    uint4 kr[kPreVecs], vr[kPreVecs];
#pragma unroll
    for (int c = 0; c < kPreVecs; ++c) {
      const int i = lane + 32 * c;
      if (i < row_vecs) {
        kr[c] = __ldg(ks + i);
        if (has_v) vr[c] = __ldg(vs + i);
      }
    }
    // sequence owning token t: largest b with cu_new[b] <= t
    int lo = 0, hi = n_seqs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu(mid) <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int start = cu(b);
    if (t < start || t >= cu(b + 1)) {  // offsets not monotone
      if (lane == 0) flag_error(err, PSW_DEVERR_LENGTH);
      continue;
    }
    const int64_t pos = static_cast<int64_t>(past_lens[b]) + (t - start);
    const int64_t page = pos / kBlockSize;
    if (pos < 0 || page >= max_blocks) {
      if (lane == 0) flag_error(err, pos < 0 ? PSW_DEVERR_LENGTH : PSW_DEVERR_CAPACITY);
      continue;
    }
    const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + page];
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) flag_error(err, PSW_DEVERR_BLOCK_ID);
      continue;
    }
    const int64_t slot = static_cast<int64_t>(blk) * kBlockSize + pos % kBlockSize;
    uint4* kd = k_pool + slot * row_vecs;
#pragma unroll
    for (int c = 0; c < kPreVecs; ++c) {
      const int i = lane + 32 * c;
      if (i < row_vecs) kd[i] = kr[c];
    }
    for (int i = lane + 32 * kPreVecs; i < row_vecs; i += 32) kd[i] = __ldg(ks + i);
    if (has_v) {
      uint4* vd = v_pool + slot * row_vecs;
#pragma unroll
      for (int c = 0; c < kPreVecs; ++c) {
        const int i = lane + 32 * c;
        if (i < row_vecs) vd[i] = vr[c];
      }
      for (int i = lane + 32 * kPreVecs; i < row_vecs; i += 32) vd[i] = __ldg(vs + i);
    }
  }
}

}  // namespace

cudaError_t launch_kv_cache_write(const LayerArgs& L, const void* k, const void* v,
                                  const int32_t* cu_new, const int32_t* past_lens, int n_seqs,
                                  const int32_t* block_table, int max_blocks, int64_t num_blocks,
                                  void* k_pool, void* v_pool, int num_sms, int32_t* err,
                                  cudaStream_t stream) {
  if (n_seqs == 0) return cudaSuccess;
  const int row_vecs = L.n_kv * L.hd * 2 / 16;
  const int grid = num_sms * 4;
  kv_cache_write_kernel<<<grid, kWarpsPerBlock * 32, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), cu_new, past_lens, n_seqs,
      block_table, max_blocks, num_blocks, row_vecs, static_cast<uint4*>(k_pool),
      static_cast<uint4*>(v_pool), err);
  return cudaGetLastError();
}

}  // namespace psw

// ---------------------------------------------------------------- FP8 pages
// The cache write into e4m3 pools: each (token, KV head) row of head_dim
// values becomes head_dim one-byte codes and one fp32 scale:
//   amax = max |x|, scale = amax / 448, code_d = e4m3(x_d * (448 / amax))
// (fp32 division and product rounded to nearest, the conversion rounding to
// nearest even and saturating at 448; an all-zero row: scale 0, codes 0).
// One warp per token; the row of one KV head at a time, 8 or 16 values per
// lane, its amax reduced with shuffles.

namespace psw {
namespace {

template <int HD>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
kv_cache_write_fp8_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                          const int32_t* __restrict__ cu_new,
                          const int32_t* __restrict__ past_lens, int n_seqs,
                          const int32_t* __restrict__ block_table, int max_blocks,
                          int64_t num_blocks, int n_kv, uint8_t* __restrict__ k_pool8,
                          uint8_t* __restrict__ v_pool8, float* __restrict__ k_scale,
                          float* __restrict__ v_scale, int32_t* err) {
  constexpr int kPer = HD / 32;  // values per lane
  __shared__ int32_t s_cu[kStagedOffsets];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool staged = n_seqs < kStagedOffsets;  // uniform over the grid
  if (staged) {
    for (int i = threadIdx.x; i <= n_seqs; i += blockDim.x) s_cu[i] = cu_new[i];
    __syncthreads();
  }
  auto cu = [&](int i) { return staged ? s_cu[i] : cu_new[i]; };
  const int total = cu(n_seqs);
  const bool has_v = v_pool8 != nullptr;
  for (int t = blockIdx.x * kWarpsPerBlock + warp; t < total;
       t += gridDim.x * kWarpsPerBlock) {
    int lo = 0, hi = n_seqs;  // sequence owning token t: largest b with cu_new[b] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu(mid) <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int start = cu(b);
    if (t < start || t >= cu(b + 1)) {  // offsets not monotone
      if (lane == 0) flag_error(err, PSW_DEVERR_LENGTH);
      continue;
    }
    const int64_t pos = static_cast<int64_t>(past_lens[b]) + (t - start);
    const int64_t page = pos / kBlockSize;
    if (pos < 0 || page >= max_blocks) {
      if (lane == 0) flag_error(err, pos < 0 ? PSW_DEVERR_LENGTH : PSW_DEVERR_CAPACITY);
      continue;
    }
    const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + page];
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) flag_error(err, PSW_DEVERR_BLOCK_ID);
      continue;
    }
    const int64_t slot = static_cast<int64_t>(blk) * kBlockSize + pos % kBlockSize;
    for (int kv = 0; kv < (has_v ? 2 : 1); ++kv) {
      const __nv_bfloat16* src = (kv == 0 ? k : v) + static_cast<int64_t>(t) * n_kv * HD;
      uint8_t* dst8 = (kv == 0 ? k_pool8 : v_pool8) + slot * n_kv * HD;
      float* dsts = (kv == 0 ? k_scale : v_scale) + slot * n_kv;
      for (int g = 0; g < n_kv; ++g) {
        float x[kPer];
        const uint4* s4 = reinterpret_cast<const uint4*>(src + g * HD) + lane * (kPer / 8);
#pragma unroll
        for (int c = 0; c < kPer / 8; ++c) {
          const uint4 u = s4[c];
          const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[c * 8 + 2 * e] = __uint_as_float(wd[e] << 16);
            x[c * 8 + 2 * e + 1] = __uint_as_float(wd[e] & 0xFFFF0000u);
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < kPer; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
        uint32_t codes[kPer / 4];
#pragma unroll
        for (int e = 0; e < kPer; e += 4) {
          const __nv_fp8x2_storage_t c01 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fmul_rn(x[e], inv), __fmul_rn(x[e + 1], inv)), __NV_SATFINITE,
              __NV_E4M3);
          const __nv_fp8x2_storage_t c23 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fmul_rn(x[e + 2], inv), __fmul_rn(x[e + 3], inv)), __NV_SATFINITE,
              __NV_E4M3);
          codes[e / 4] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
        }
        uint8_t* d = dst8 + g * HD + lane * kPer;
        if constexpr (kPer == 8)
          *reinterpret_cast<uint2*>(d) = make_uint2(codes[0], codes[1]);
        else
          *reinterpret_cast<uint4*>(d) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        if (lane == 0) dsts[g] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_cache_write_fp8(const LayerArgs& L, const void* k, const void* v,
                                      const int32_t* cu_new, const int32_t* past_lens,
                                      int n_seqs, const int32_t* block_table, int max_blocks,
                                      int64_t num_blocks, void* k_pool8, void* v_pool8,
                                      float* k_scale, float* v_scale, int num_sms, int32_t* err,
                                      cudaStream_t stream) {
  if (n_seqs == 0) return cudaSuccess;
  const int grid = num_sms * 4;
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* k8 = static_cast<uint8_t*>(k_pool8);
  auto* v8 = static_cast<uint8_t*>(v_pool8);
  if (L.hd == 256)
    kv_cache_write_fp8_kernel<256><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        kb, vb, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, L.n_kv, k8, v8,
        k_scale, v_scale, err);
  else
    kv_cache_write_fp8_kernel<512><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        kb, vb, cu_new, past_lens, n_seqs, block_table, max_blocks, num_blocks, L.n_kv, k8, v8,
        k_scale, v_scale, err);
  return cudaGetLastError();
}

}  // namespace psw
