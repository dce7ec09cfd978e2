// psw_internal.h -- host-side launchers shared between the API translation
// unit and the kernel translation units of libpsw. Library-internal.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/psw.h"

namespace psw {

constexpr int kBlockSize = 16;          // tokens per page
constexpr int kMaxDecodeCtas = 512;     // upper bound on the persistent decode grid
constexpr int kQHeadsPerUnit = 8;       // query heads handled together per KV head
constexpr int kDecodePlanAlign = 256;
// The first kWsCounterBytes of every workspace hold counters that each call
// leaves at zero (the decode merge tickets, one int32 per CTA); the caller
// zero-fills a workspace once before its first use (PSW_WORKSPACE_COUNTER_BYTES).
constexpr size_t kWsCounterBytes = PSW_WORKSPACE_COUNTER_BYTES;
static_assert(kMaxDecodeCtas * 4 <= PSW_WORKSPACE_COUNTER_BYTES, "one ticket per decode CTA");

struct LayerArgs {
  int n_q, n_kv, hd, window;
  float softcap, scale;
  bool k_eq_v;
  int group() const { return n_q / n_kv; }
  int qchunks() const { return (group() + kQHeadsPerUnit - 1) / kQHeadsPerUnit; }
};

struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
};

// Host checks of attn_decode_paged's arguments other than the workspace, in
// the order that call reports them (layer, pointers, V pool, pages, n_seqs,
// alignment). Fills *L on success. Returns a PSW_* code.
int check_decode_args(const psw_layer_t* layer, const void* q, const void* k_pool,
                      const void* v_pool, const psw_pages_t* pages, const int32_t* seq_lens,
                      int32_t n_seqs, const float* out, LayerArgs* L);

// Current device's properties (cached per device).
cudaError_t device_info(DeviceInfo* info);

// Per-device error word used by every kernel (device pointer).
int32_t* device_error_word();

// Sets a kernel's dynamic shared-memory limit on the current device, once per
// (kernel, device); safe to call from several host threads. Returns a PSW_* code.
int set_smem_limit(const void* kernel, int bytes);

// Testing hook set by psw_testing_stall: the CTA whose producer leaves tile
// copy `tile` (counted from 0 over its own copies) unissued; -1: none.
struct StallHook {
  int cta = -1, tile = -1;
};
constexpr int kStallDecode = 1, kStallPrefill = 2;
StallHook stall_hook(int kernel);

// Decode workspace layout (bytes): merge tickets (counter block) | partial O |
// partial (m, l).
struct DecodeWorkspace {
  size_t o_bytes, ml_bytes, ticket_bytes, total;
  size_t o_offset, ml_offset, ticket_offset;
};
DecodeWorkspace decode_workspace_layout(const LayerArgs& L, int n_seqs, int max_ctas);

cudaError_t launch_kv_cache_write(const LayerArgs& L, const void* k, const void* v,
                                  const int32_t* cu_new, const int32_t* past_lens, int n_seqs,
                                  const int32_t* block_table, int max_blocks, int64_t num_blocks,
                                  void* k_pool, void* v_pool, int num_sms, int32_t* err,
                                  cudaStream_t stream);

// Append mode of the decode (attn_decode_paged_append): the step's new K/V
// row of each sequence (k_new / v_new [n_seqs][n_kv][hd] bf16) is written to
// its slot at position seq_len - 1 of the pools and used in place of that
// slot's staged copy. All NULL: plain decode.
struct AppendArgs {
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  void* k_pool = nullptr;
  void* v_pool = nullptr;
};

// Returns a PSW_* code. With k_scale (FP8 pages), the maps are e4m3 pool maps
// (make_pool_tensor_map_fp8) and k_scale / v_scale the per-row scales
// (v_scale unused with k_eq_v). `append` is for bf16 pages only.
int launch_decode(const LayerArgs& L, const void* q, const CUtensorMap& k_map,
                  const CUtensorMap& v_map, const int32_t* block_table, int max_blocks,
                  int64_t num_blocks, const int32_t* seq_lens, int n_seqs, float* out, float* lse,
                  void* ws, size_t ws_bytes, int num_sms, int32_t* err, cudaStream_t stream,
                  const float* k_scale = nullptr, const float* v_scale = nullptr,
                  AppendArgs append = AppendArgs{});

// TMA descriptor of an e4m3 pool [num_blocks][16][n_kv][hd] (one byte per
// value) seen as [slot][chunk of 64 codes][64], box = 16 slots x 1 chunk.
int make_pool_tensor_map_fp8(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv,
                             int hd);

// FP8 cache write: each (token, KV head) row quantised to e4m3 with one fp32
// scale (amax / 448). v / v_pool8 / v_scale NULL with k_eq_v.
cudaError_t launch_kv_cache_write_fp8(const LayerArgs& L, const void* k, const void* v,
                                      const int32_t* cu_new, const int32_t* past_lens,
                                      int n_seqs, const int32_t* block_table, int max_blocks,
                                      int64_t num_blocks, void* k_pool8, void* v_pool8,
                                      float* k_scale, float* v_scale, int num_sms, int32_t* err,
                                      cudaStream_t stream);

// Pre-attention step parameters after validation.
struct NormRopeArgs {
  float theta, eps;
  int rope_angles;  // rotated pairs: floor(partial_rotary_factor * head_dim / 2)
  const float *q_weight, *k_weight, *v_weight;
};

// Per-head RMS-norm of q (and k, v when given), proportional RoPE of q and
// k, q into q_out and k / v into their pages. Returns a PSW_* code.
int launch_qkv_norm_rope(const LayerArgs& L, const NormRopeArgs& R, const void* q, const void* k,
                         const void* v, const int32_t* cu_new, const int32_t* past_lens,
                         int n_seqs, const int32_t* block_table, int max_blocks,
                         int64_t num_blocks, void* q_out, void* k_pool, void* v_pool, int num_sms,
                         int32_t* err, cudaStream_t stream);

// Prefill workspace: a work list of the (sequence, block) units.
size_t prefill_workspace_bytes(const LayerArgs& L, int n_seqs, int max_q_len);

// Returns a PSW_* code.
int launch_prefill(const LayerArgs& L, const CUtensorMap& q_map, const CUtensorMap& k_map,
                   const CUtensorMap& v_map, const int32_t* cu_q, const int32_t* past_lens,
                   int n_seqs, int n_q_total, int max_q_len, const int32_t* block_table,
                   int max_blocks, int64_t num_blocks, float* out, float* lse, void* ws,
                   int num_sms, int32_t* err, cudaStream_t stream);

// TMA descriptor of q [n_q_total][n_q][hd] with one box = 64 columns x G
// heads x (128 / G) tokens, 128-byte swizzle.
int make_query_tensor_map(CUtensorMap* map, const void* q, int n_q_total, int n_q, int hd,
                          int group);

// Builds the TMA descriptor of a pool seen as [slot][chunk of 64 elems][64]
// with one box = 16 slots x 1 chunk, 128-byte swizzle.
int make_pool_tensor_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv,
                         int hd);
// Pool view whose box is box_slots slots (a page or half of one) of box_chunks
// 64-element chunks of one KV head, landing in shared memory as
// [chunk][box_slots rows][128 B].
int make_pool_page_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv, int hd,
                       int box_slots, int box_chunks);

}  // namespace psw
