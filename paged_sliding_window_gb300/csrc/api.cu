// api.cu -- the extern "C" surface of libpsw (include/psw.h): argument
// validation (every error is returned before anything is launched), TMA
// descriptors for the page pools, the per-device error word, and dispatch to
// the kernel launchers.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "psw_internal.h"

namespace psw {

// Device-side error word: kernels OR PSW_DEVERR_* bits into it.
__device__ int32_t g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  DeviceInfo info{};
  int32_t* err = nullptr;
};
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

DeviceState* current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_devices[dev];
  if (!st.ready) {
    DeviceInfo info{};
    info.device = dev;
    if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess)
      return nullptr;
    void* err = nullptr;
    if (cudaGetSymbolAddress(&err, g_error_word) != cudaSuccess) return nullptr;
    st.info = info;
    st.err = static_cast<int32_t*>(err);
    st.ready = true;
  }
  return &st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layer(const psw_layer_t* layer, LayerArgs* out) {
  if (layer == nullptr) return PSW_ENULL;
  if (layer->n_q_heads <= 0 || layer->n_kv_heads <= 0 ||
      layer->n_q_heads % layer->n_kv_heads != 0)
    return PSW_EINVAL_HEADS;
  if (layer->head_dim != 256 && layer->head_dim != 512) return PSW_EINVAL_HDIM;
  if (!(layer->softcap >= 0.f) || !isfinite(layer->softcap)) return PSW_EINVAL_SOFTCAP;
  if (layer->window < 0) return PSW_EINVAL_WINDOW;
  if (layer->block_size != kBlockSize) return PSW_EINVAL_BLOCKSIZE;
  if (!(layer->scale > 0.f) || !isfinite(layer->scale)) return PSW_EINVAL_SCALE;
  if (layer->k_eq_v != 0 && layer->k_eq_v != 1) return PSW_EINVAL_KEQV;
  out->n_q = layer->n_q_heads;
  out->n_kv = layer->n_kv_heads;
  out->hd = layer->head_dim;
  out->window = layer->window;
  out->softcap = layer->softcap;
  out->scale = layer->scale;
  out->k_eq_v = layer->k_eq_v != 0;
  return PSW_OK;
}

int check_pages(const psw_pages_t* pages) {
  if (pages == nullptr || pages->block_table == nullptr) return PSW_ENULL;
  if (pages->max_blocks_per_seq <= 0 || pages->num_blocks <= 0) return PSW_ECAPACITY;
  // block ids are int32 and TMA slot coordinates (id * 16) must fit int32
  if (pages->num_blocks > (int64_t{1} << 27)) return PSW_ECAPACITY;
  if (static_cast<int64_t>(pages->max_blocks_per_seq) * kBlockSize > INT32_MAX)
    return PSW_ECAPACITY;
  return PSW_OK;
}

// k_eq_v: V must be absent; otherwise present.
int check_v(const LayerArgs& L, const void* v_ptr) {
  if (L.k_eq_v && v_ptr != nullptr) return PSW_EINVAL_KEQV;
  if (!L.k_eq_v && v_ptr == nullptr) return PSW_EINVAL_KEQV;
  return PSW_OK;
}

int device_ready(DeviceState** st) {
  *st = current_device();
  if (*st == nullptr) return PSW_EDEVICE;
  if ((*st)->info.cc_major != 10 || (*st)->info.cc_minor != 3) return PSW_EDEVICE;
  return PSW_OK;
}

struct SmemLimitSet {
  const void* kernel;
  int device;
};
std::mutex g_attr_mutex;
SmemLimitSet g_attr_done[256];
int g_attr_count = 0;

}  // namespace

int set_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PSW_EDEVICE;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  for (int i = 0; i < g_attr_count; ++i)
    if (g_attr_done[i].kernel == kernel && g_attr_done[i].device == dev) return PSW_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return PSW_ELAUNCH;
  // a full table only means the attribute is set again on later calls
  if (g_attr_count < static_cast<int>(sizeof(g_attr_done) / sizeof(g_attr_done[0])))
    g_attr_done[g_attr_count++] = SmemLimitSet{kernel, dev};
  return PSW_OK;
}

namespace {
std::mutex g_stall_mutex;
int g_stall_kernel = 0;
StallHook g_stall;
}  // namespace

StallHook stall_hook(int kernel) {
  std::lock_guard<std::mutex> lock(g_stall_mutex);
  return g_stall_kernel == kernel ? g_stall : StallHook{};
}

int check_decode_args(const psw_layer_t* layer, const void* q, const void* k_pool,
                      const void* v_pool, const psw_pages_t* pages, const int32_t* seq_lens,
                      int32_t n_seqs, const float* out, LayerArgs* L) {
  int rc = check_layer(layer, L);
  if (rc != PSW_OK) return rc;
  if (q == nullptr || k_pool == nullptr || seq_lens == nullptr || out == nullptr)
    return PSW_ENULL;
  if ((rc = check_v(*L, v_pool)) != PSW_OK) return rc;
  if ((rc = check_pages(pages)) != PSW_OK) return rc;
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PSW_EALIGN;
  return PSW_OK;
}

cudaError_t device_info(DeviceInfo* info) {
  DeviceState* st = current_device();
  if (st == nullptr) return cudaErrorNoDevice;
  *info = st->info;
  return cudaSuccess;
}

int32_t* device_error_word() {
  DeviceState* st = current_device();
  return st ? st->err : nullptr;
}

int make_pool_tensor_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv,
                         int hd) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PSW_ETENSORMAP;
  // [slot][chunk of 64 elements across (kv head, head_dim)][64 elements]
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(n_kv) * (hd / 64),
                              static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(n_kv) * hd * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[3] = {1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PSW_OK : PSW_ETENSORMAP;
}

int make_pool_page_map(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv, int hd,
                       int box_slots, int box_chunks) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PSW_ETENSORMAP;
  // [chunk of 64 elements across (kv head, head_dim)][slot][64 elements]: one
  // box is box_slots slots (a page, or half of one) of box_chunks chunks and
  // lands in shared memory as [chunk][box_slots rows][128 B]
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_blocks) * kBlockSize,
                              static_cast<cuuint64_t>(n_kv) * (hd / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(n_kv) * hd * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_slots),
                             static_cast<cuuint32_t>(box_chunks)};
  const cuuint32_t estr[3] = {1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PSW_OK : PSW_ETENSORMAP;
}

int make_pool_tensor_map_fp8(CUtensorMap* map, const void* pool, int64_t num_blocks, int n_kv,
                             int hd) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PSW_ETENSORMAP;
  // [slot][chunk of 64 codes across (kv head, head_dim)][64 codes]; a box is
  // 16 slots x 1 chunk = 1 KB, unswizzled (the consumers convert it with
  // plain loads)
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(n_kv) * (hd / 64),
                              static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  const cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(n_kv) * hd};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[3] = {1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PSW_OK : PSW_ETENSORMAP;
}

int make_query_tensor_map(CUtensorMap* map, const void* q, int n_q_total, int n_q, int hd,
                          int group) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PSW_ETENSORMAP;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(n_q),
                              static_cast<cuuint64_t>(n_q_total)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2,
                                 static_cast<cuuint64_t>(n_q) * hd * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(128 / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PSW_OK : PSW_ETENSORMAP;
}

}  // namespace psw

using namespace psw;

extern "C" {

int psw_workspace_bytes(const psw_layer_t* layer, int32_t n_seqs, int32_t max_seq_len,
                        size_t* bytes) {
  LayerArgs L;
  int rc = check_layer(layer, &L);
  if (rc != PSW_OK) return rc;
  if (bytes == nullptr) return PSW_ENULL;
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (max_seq_len < 0) return PSW_ECAPACITY;
  const size_t dec = decode_workspace_layout(L, n_seqs, kMaxDecodeCtas).total;
  const size_t pre = prefill_workspace_bytes(L, n_seqs, max_seq_len);
  *bytes = dec > pre ? dec : pre;
  return PSW_OK;
}

int kv_cache_write(const psw_layer_t* layer, const void* k, const void* v,
                   const int32_t* cu_new, const int32_t* past_lens, int32_t n_seqs,
                   const psw_pages_t* pages, void* k_pool, void* v_pool, psw_stream_t stream) {
  LayerArgs L;
  int rc = check_layer(layer, &L);
  if (rc != PSW_OK) return rc;
  if (k == nullptr || cu_new == nullptr || past_lens == nullptr || k_pool == nullptr)
    return PSW_ENULL;
  if ((rc = check_v(L, v)) != PSW_OK) return rc;
  if ((rc = check_v(L, v_pool)) != PSW_OK) return rc;
  if ((rc = check_pages(pages)) != PSW_OK) return rc;
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PSW_EALIGN;
  if (n_seqs == 0) return PSW_OK;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  cudaError_t e = launch_kv_cache_write(L, k, v, cu_new, past_lens, n_seqs, pages->block_table,
                                        pages->max_blocks_per_seq, pages->num_blocks, k_pool,
                                        v_pool, st->info.num_sms, st->err,
                                        reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

int attn_decode_paged(const psw_layer_t* layer, const void* q, const void* k_pool,
                      const void* v_pool, const psw_pages_t* pages, const int32_t* seq_lens,
                      int32_t n_seqs, float* out, float* lse, void* ws, size_t ws_bytes,
                      psw_stream_t stream) {
  LayerArgs L;
  int rc = check_decode_args(layer, q, k_pool, v_pool, pages, seq_lens, n_seqs, out, &L);
  if (rc != PSW_OK) return rc;
  if (n_seqs == 0) return PSW_OK;
  if (ws == nullptr) return PSW_EWORKSPACE;
  if (ws_bytes < decode_workspace_layout(L, n_seqs, kMaxDecodeCtas).total) return PSW_EWORKSPACE;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  CUtensorMap k_map, v_map;
  if ((rc = make_pool_tensor_map(&k_map, k_pool, pages->num_blocks, L.n_kv, L.hd)) != PSW_OK)
    return rc;
  if (L.k_eq_v) {
    v_map = k_map;
  } else if ((rc = make_pool_tensor_map(&v_map, v_pool, pages->num_blocks, L.n_kv, L.hd)) !=
             PSW_OK) {
    return rc;
  }
  return launch_decode(L, q, k_map, v_map, pages->block_table, pages->max_blocks_per_seq,
                       pages->num_blocks, seq_lens, n_seqs, out, lse, ws, ws_bytes,
                       st->info.num_sms, st->err, reinterpret_cast<cudaStream_t>(stream));
}

int attn_decode_paged_append(const psw_layer_t* layer, const void* q, const void* k_new,
                             const void* v_new, void* k_pool, void* v_pool,
                             const psw_pages_t* pages, const int32_t* seq_lens, int32_t n_seqs,
                             float* out, float* lse, void* ws, size_t ws_bytes,
                             psw_stream_t stream) {
  LayerArgs L;
  int rc = check_decode_args(layer, q, k_pool, v_pool, pages, seq_lens, n_seqs, out, &L);
  if (rc != PSW_OK) return rc;
  if (k_new == nullptr) return PSW_ENULL;
  if ((rc = check_v(L, v_new)) != PSW_OK) return rc;
  if (!aligned16(k_new) || !aligned16(v_new)) return PSW_EALIGN;
  if (n_seqs == 0) return PSW_OK;
  if (ws == nullptr) return PSW_EWORKSPACE;
  if (ws_bytes < decode_workspace_layout(L, n_seqs, kMaxDecodeCtas).total) return PSW_EWORKSPACE;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  CUtensorMap k_map, v_map;
  if ((rc = make_pool_tensor_map(&k_map, k_pool, pages->num_blocks, L.n_kv, L.hd)) != PSW_OK)
    return rc;
  if (L.k_eq_v) {
    v_map = k_map;
  } else if ((rc = make_pool_tensor_map(&v_map, v_pool, pages->num_blocks, L.n_kv, L.hd)) !=
             PSW_OK) {
    return rc;
  }
  AppendArgs app;
  app.k_new = k_new;
  app.v_new = v_new;
  app.k_pool = k_pool;
  app.v_pool = v_pool;
  return launch_decode(L, q, k_map, v_map, pages->block_table, pages->max_blocks_per_seq,
                       pages->num_blocks, seq_lens, n_seqs, out, lse, ws, ws_bytes,
                       st->info.num_sms, st->err, reinterpret_cast<cudaStream_t>(stream),
                       nullptr, nullptr, app);
}

namespace {
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
}  // namespace

int kv_cache_write_fp8(const psw_layer_t* layer, const void* k, const void* v,
                       const int32_t* cu_new, const int32_t* past_lens, int32_t n_seqs,
                       const psw_pages_t* pages, void* k_pool8, void* v_pool8, float* k_scale,
                       float* v_scale, psw_stream_t stream) {
  LayerArgs L;
  int rc = check_layer(layer, &L);
  if (rc != PSW_OK) return rc;
  if (k == nullptr || cu_new == nullptr || past_lens == nullptr || k_pool8 == nullptr ||
      k_scale == nullptr)
    return PSW_ENULL;
  if ((rc = check_v(L, v)) != PSW_OK) return rc;
  if ((rc = check_v(L, v_pool8)) != PSW_OK) return rc;
  if ((rc = check_v(L, v_scale)) != PSW_OK) return rc;
  if ((rc = check_pages(pages)) != PSW_OK) return rc;
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool8) || !aligned16(v_pool8) ||
      !aligned4(k_scale) || !aligned4(v_scale))
    return PSW_EALIGN;
  if (n_seqs == 0) return PSW_OK;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  cudaError_t e = launch_kv_cache_write_fp8(
      L, k, v, cu_new, past_lens, n_seqs, pages->block_table, pages->max_blocks_per_seq,
      pages->num_blocks, k_pool8, v_pool8, k_scale, v_scale, st->info.num_sms, st->err,
      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PSW_OK : PSW_ELAUNCH;
}

int attn_decode_paged_fp8(const psw_layer_t* layer, const void* q, const void* k_pool8,
                          const void* v_pool8, const float* k_scale, const float* v_scale,
                          const psw_pages_t* pages, const int32_t* seq_lens, int32_t n_seqs,
                          float* out, float* lse, void* ws, size_t ws_bytes,
                          psw_stream_t stream) {
  LayerArgs L;
  int rc = check_decode_args(layer, q, k_pool8, v_pool8, pages, seq_lens, n_seqs, out, &L);
  if (rc != PSW_OK) return rc;
  if (k_scale == nullptr) return PSW_ENULL;
  if ((rc = check_v(L, v_scale)) != PSW_OK) return rc;
  if (!aligned4(k_scale) || !aligned4(v_scale)) return PSW_EALIGN;
  if (n_seqs == 0) return PSW_OK;
  if (ws == nullptr) return PSW_EWORKSPACE;
  if (ws_bytes < decode_workspace_layout(L, n_seqs, kMaxDecodeCtas).total) return PSW_EWORKSPACE;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  CUtensorMap k_map, v_map;
  if ((rc = make_pool_tensor_map_fp8(&k_map, k_pool8, pages->num_blocks, L.n_kv, L.hd)) !=
      PSW_OK)
    return rc;
  if (L.k_eq_v) {
    v_map = k_map;
  } else if ((rc = make_pool_tensor_map_fp8(&v_map, v_pool8, pages->num_blocks, L.n_kv,
                                            L.hd)) != PSW_OK) {
    return rc;
  }
  return launch_decode(L, q, k_map, v_map, pages->block_table, pages->max_blocks_per_seq,
                       pages->num_blocks, seq_lens, n_seqs, out, lse, ws, ws_bytes,
                       st->info.num_sms, st->err, reinterpret_cast<cudaStream_t>(stream),
                       k_scale, L.k_eq_v ? k_scale : v_scale);
}

int attn_prefill_chunked(const psw_layer_t* layer, const void* q, const int32_t* cu_q,
                         const int32_t* past_lens, int32_t n_seqs, int32_t n_q_total,
                         int32_t max_q_len, const void* k_pool, const void* v_pool,
                         const psw_pages_t* pages, float* out, float* lse, void* ws,
                         size_t ws_bytes, psw_stream_t stream) {
  LayerArgs L;
  int rc = check_layer(layer, &L);
  if (rc != PSW_OK) return rc;
  if (q == nullptr || cu_q == nullptr || past_lens == nullptr || k_pool == nullptr ||
      out == nullptr)
    return PSW_ENULL;
  if ((rc = check_v(L, v_pool)) != PSW_OK) return rc;
  if ((rc = check_pages(pages)) != PSW_OK) return rc;
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (L.group() > 128) return PSW_EINVAL_HEADS;
  if (max_q_len < 0 || n_q_total < 0) return PSW_ECAPACITY;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PSW_EALIGN;
  if (n_seqs == 0 || max_q_len == 0 || n_q_total == 0) return PSW_OK;
  if (n_seqs > 65535) return PSW_EINVAL_NSEQS;
  // work items (sequence, block of 128 / G tokens, KV head, head_dim half) must
  // be countable in 32 bits
  const int64_t blocks = (static_cast<int64_t>(max_q_len) + 128 / L.group() - 1) / (128 / L.group());
  if (static_cast<int64_t>(n_seqs) * blocks * L.n_kv * (L.hd / 256) > 0x7fffffffLL)
    return PSW_ECAPACITY;
  if (ws == nullptr || ws_bytes < prefill_workspace_bytes(L, n_seqs, max_q_len))
    return PSW_EWORKSPACE;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  CUtensorMap q_map, k_map, v_map;
  if ((rc = make_query_tensor_map(&q_map, q, n_q_total, L.n_q, L.hd, L.group())) != PSW_OK)
    return rc;
  // K: half-page boxes over every chunk of a head ([chunk][8 rows][128 B]),
  // or over one head_dim half at head_dim 512 with k_eq_v;
  // V: whole-page boxes of four chunks ([chunk][16 rows][128 B])
  const int k_box_chunks = (L.hd == 512 && L.k_eq_v) ? 4 : L.hd / 64;
  if ((rc = make_pool_page_map(&k_map, k_pool, pages->num_blocks, L.n_kv, L.hd, kBlockSize / 2,
                               k_box_chunks)) != PSW_OK)
    return rc;
  if (L.k_eq_v) {
    v_map = k_map;
  } else if ((rc = make_pool_page_map(&v_map, v_pool, pages->num_blocks, L.n_kv, L.hd,
                                      kBlockSize, 4)) != PSW_OK) {
    return rc;
  }
  return launch_prefill(L, q_map, k_map, v_map, cu_q, past_lens, n_seqs, n_q_total, max_q_len,
                        pages->block_table, pages->max_blocks_per_seq, pages->num_blocks, out,
                        lse, ws, st->info.num_sms, st->err,
                        reinterpret_cast<cudaStream_t>(stream));
}

int qkv_norm_rope_cache_write(const psw_layer_t* layer, const psw_norm_rope_t* rn,
                              const void* q, const void* k, const void* v,
                              const int32_t* cu_new, const int32_t* past_lens, int32_t n_seqs,
                              const psw_pages_t* pages, void* q_out, void* k_pool, void* v_pool,
                              psw_stream_t stream) {
  LayerArgs L;
  int rc = check_layer(layer, &L);
  if (rc != PSW_OK) return rc;
  if (rn == nullptr || q == nullptr || q_out == nullptr || cu_new == nullptr ||
      past_lens == nullptr)
    return PSW_ENULL;
  if (!(rn->theta > 0.f) || !isfinite(rn->theta) || !(rn->partial_rotary_factor > 0.f) ||
      !(rn->partial_rotary_factor <= 1.f) || !(rn->eps >= 0.f) || !isfinite(rn->eps))
    return PSW_EINVAL_ROPE;
  const bool cache = k != nullptr;
  if (cache) {
    if (k_pool == nullptr) return PSW_ENULL;
    if ((rc = check_v(L, v)) != PSW_OK) return rc;
    if ((rc = check_v(L, v_pool)) != PSW_OK) return rc;
    if ((rc = check_pages(pages)) != PSW_OK) return rc;
  } else if (v != nullptr || k_pool != nullptr || v_pool != nullptr) {
    return PSW_ENULL;  // a q-only call names no K/V rows and no pools
  }
  if (n_seqs < 0) return PSW_EINVAL_NSEQS;
  if (!aligned16(q) || !aligned16(q_out) || !aligned16(k) || !aligned16(v) ||
      !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(rn->q_weight) ||
      !aligned16(rn->k_weight) || !aligned16(rn->v_weight))
    return PSW_EALIGN;
  if (n_seqs == 0) return PSW_OK;
  DeviceState* st;
  if ((rc = device_ready(&st)) != PSW_OK) return rc;
  NormRopeArgs R;
  R.theta = rn->theta;
  R.eps = rn->eps;
  R.rope_angles = static_cast<int>(rn->partial_rotary_factor * static_cast<float>(L.hd) / 2.f);
  if (R.rope_angles > L.hd / 2) R.rope_angles = L.hd / 2;
  R.q_weight = rn->q_weight;
  R.k_weight = rn->k_weight;
  R.v_weight = rn->v_weight;
  return launch_qkv_norm_rope(L, R, q, k, v, cu_new, past_lens, n_seqs,
                              cache ? pages->block_table : nullptr,
                              cache ? pages->max_blocks_per_seq : 0,
                              cache ? pages->num_blocks : 0, q_out, k_pool, v_pool,
                              st->info.num_sms, st->err, reinterpret_cast<cudaStream_t>(stream));
}

int psw_kv_share_map(int32_t n_layers, int32_t pattern, int32_t n_shared, int32_t* is_full,
                     int32_t* target) {
  if (n_layers <= 0 || pattern <= 0 || n_shared < 0 || n_shared >= n_layers)
    return PSW_EINVAL_LAYERS;
  const int32_t owners = n_layers - n_shared;
  // last cache-owning layer of each type (-1: none)
  int32_t last_owner[2] = {-1, -1};
  for (int32_t i = 0; i < owners; ++i) last_owner[(i + 1) % pattern == 0 ? 1 : 0] = i;
  for (int32_t i = owners; i < n_layers; ++i)
    if (last_owner[(i + 1) % pattern == 0 ? 1 : 0] < 0) return PSW_EINVAL_LAYERS;
  for (int32_t i = 0; i < n_layers; ++i) {
    const int full = (i + 1) % pattern == 0 ? 1 : 0;
    if (is_full != nullptr) is_full[i] = full;
    if (target != nullptr) target[i] = i < owners ? i : last_owner[full];
  }
  return PSW_OK;
}

int psw_testing_stall(int32_t kernel, int32_t cta, int32_t tile) {
  if (kernel < 0 || kernel > kStallPrefill) return PSW_EINVAL_NSEQS;
  if (kernel != 0 && (cta < 0 || tile < 0)) return PSW_EINVAL_NSEQS;
  std::lock_guard<std::mutex> lock(g_stall_mutex);
  g_stall_kernel = kernel;
  g_stall = kernel == 0 ? StallHook{} : StallHook{cta, tile};
  return PSW_OK;
}

int psw_get_error(psw_stream_t stream, int32_t* device_error_out) {
  if (device_error_out == nullptr) return PSW_ENULL;
  DeviceState* st = current_device();
  if (st == nullptr) return PSW_EDEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PSW_ELAUNCH;
  int32_t v = 0;
  if (cudaMemcpy(&v, st->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PSW_ELAUNCH;
  const int32_t zero = 0;
  if (cudaMemcpy(st->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return PSW_ELAUNCH;
  *device_error_out = v;
  return PSW_OK;
}

const char* psw_strerror(int code) {
  switch (code) {
    case PSW_OK: return "ok";
    case PSW_ENULL: return "a required pointer is NULL";
    case PSW_EINVAL_HEADS: return "n_q_heads must be a positive multiple of n_kv_heads";
    case PSW_EINVAL_HDIM: return "head_dim must be 256 or 512";
    case PSW_EINVAL_SOFTCAP: return "softcap must be finite and >= 0 (0 = off)";
    case PSW_EINVAL_WINDOW: return "window must be >= 0 (0 = full attention)";
    case PSW_EINVAL_BLOCKSIZE: return "block_size must be 16";
    case PSW_EINVAL_KEQV: return "k_eq_v requires NULL V pointers; otherwise V is required";
    case PSW_EINVAL_SCALE: return "scale must be finite and > 0";
    case PSW_EINVAL_NSEQS: return "n_seqs must be >= 0";
    case PSW_EWORKSPACE: return "workspace is missing or smaller than psw_workspace_bytes()";
    case PSW_ECAPACITY: return "page table capacity out of range";
    case PSW_EALIGN: return "bf16 inputs, pools and out must be 16-byte aligned";
    case PSW_EDEVICE: return "no usable sm_103 (GB300) device";
    case PSW_ELAUNCH: return "CUDA launch failed";
    case PSW_ETENSORMAP: return "could not build the TMA descriptor of a pool";
    case PSW_ESCRATCH:
      return "batch needs more scratch than the static buffer of attn_decode_paged_noalloc";
    case PSW_ENOBLOCKS: return "the block pool has fewer free blocks than asked for";
    case PSW_EBLOCK: return "block id outside the pool, or freed more often than it is held";
    case PSW_EINVAL_LAYERS:
      return "n_layers and pattern must be > 0, n_shared in [0, n_layers), and every shared "
             "layer needs a cache-owning layer of its type";
    case PSW_EINVAL_ROPE:
      return "theta must be > 0, partial_rotary_factor in (0, 1], eps >= 0, all finite";
    default: return "unknown error";
  }
}

}  // extern "C"
