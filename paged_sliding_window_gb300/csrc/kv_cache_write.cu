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
