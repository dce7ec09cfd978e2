// decode_noalloc.cu -- paged decode for callers that cannot allocate device memory.
//
// attn_decode_paged needs a caller-provided workspace for its split-KV
// partial results. Some callers cannot hand one over: code whose device memory
// is owned entirely by another allocator with a fixed budget (a framework's
// caching allocator, an embedded runtime), or a latency-critical serving loop
// that must not call cudaMalloc after start-up, because an allocation can
// synchronise the device or fail under fragmentation. attn_decode_paged_noalloc
// gives them the same decode with the scratch taken from a buffer that is part
// of the library image itself.
//
// The buffer is a file-scope __device__ array of PSW_NOALLOC_SCRATCH_BYTES.
// The kernels only need its device address, which host code cannot take from
// the array's name (on the host that name is a stand-in, not a device
// address), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and keeps it for later
// calls. Under CUDA's lazy module loading (the default since CUDA 12.2) this
// lookup is also the moment the driver loads this translation unit's module
// and reserves the array on the device; with eager loading it was reserved
// when the library was loaded. Either way the memory then stays reserved on
// that device until the process exits. The set-up can therefore fail when the
// device is out of memory, and it must not happen inside a stream capture: a
// caller makes one call at start-up (n_seqs = 0 with valid pointers is enough;
// it does the set-up and launches nothing).
//
// All calls share the one buffer and it keeps whatever the last call left in
// it. Its first PSW_WORKSPACE_COUNTER_BYTES hold the decode merge tickets,
// which start at zero (static storage is zero-initialised) and which every
// call leaves at zero; everything else is written before it is read within a
// call. Calls whose kernels could overlap on the GPU (other streams, or other
// host threads on the same device) race on the buffer and must be serialised
// by the caller.
//
// No cudaMalloc, cudaFree or any allocating routine is called here.
#include <mutex>

#include "psw_internal.h"

namespace psw {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PSW_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxNoAllocDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxNoAllocDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices)
    return PSW_EDEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PSW_EDEVICE;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PSW_OK;
}
}  // namespace

}  // namespace psw

extern "C" int attn_decode_paged_noalloc(const psw_layer_t* layer, const void* q,
                                         const void* k_pool, const void* v_pool,
                                         const psw_pages_t* pages, const int32_t* seq_lens,
                                         int32_t n_seqs, float* out, float* lse,
                                         psw_stream_t stream) {
  // the argument errors of attn_decode_paged come first, in its order
  psw::LayerArgs L;
  int rc = psw::check_decode_args(layer, q, k_pool, v_pool, pages, seq_lens, n_seqs, out, &L);
  if (rc != PSW_OK) return rc;
  size_t need = 0;
  if ((rc = psw_workspace_bytes(layer, n_seqs, 0, &need)) != PSW_OK) return rc;
  if (need > static_cast<size_t>(PSW_NOALLOC_SCRATCH_BYTES)) return PSW_ESCRATCH;
  void* scratch = nullptr;
  if ((rc = psw::noalloc_scratch(&scratch)) != PSW_OK) return rc;
  if (n_seqs == 0) return PSW_OK;  // set-up only
  return attn_decode_paged(layer, q, k_pool, v_pool, pages, seq_lens, n_seqs, out, lse, scratch,
                           static_cast<size_t>(PSW_NOALLOC_SCRATCH_BYTES), stream);
}
