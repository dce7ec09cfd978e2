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

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
kv_cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                      const int32_t* __restrict__ cu_new, const int32_t* __restrict__ past_lens,
                      int n_seqs, const int32_t* __restrict__ block_table, int max_blocks,
                      int64_t num_blocks, int row_vecs, uint4* __restrict__ k_pool,
                      uint4* __restrict__ v_pool, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total = cu_new[n_seqs];
  for (int t = blockIdx.x * kWarpsPerBlock + warp; t < total;
       t += gridDim.x * kWarpsPerBlock) {
    // sequence owning token t: largest b with cu_new[b] <= t
    int lo = 0, hi = n_seqs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_new[mid] <= t) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int start = cu_new[b];
    if (t < start || t >= cu_new[b + 1]) {  // offsets not monotone
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
    const uint4* ks = k + static_cast<int64_t>(t) * row_vecs;
    uint4* kd = k_pool + slot * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) kd[i] = __ldg(ks + i);
    if (v_pool != nullptr) {
      const uint4* vs = v + static_cast<int64_t>(t) * row_vecs;
      uint4* vd = v_pool + slot * row_vecs;
      for (int i = lane; i < row_vecs; i += 32) vd[i] = __ldg(vs + i);
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
