/*
 * psw.h -- C ABI of the paged sliding-window attention library (libpsw.so).
 *
 * Three operations make one serving step of one attention layer of a
 * Gemma-style hybrid decoder whose KV cache lives in 16-token pages:
 *
 *   kv_cache_write        write the step's new K/V rows into their pages
 *   attn_decode_paged     one query per sequence over its paged keys
 *   attn_prefill_chunked  a chunk of queries per sequence over its paged keys
 *
 * Page layout (vLLM paged attention as described in "Gemma 4 model
 * architecture analysis" (vLLM-Kunlun), sections 6.2-6.5): a pool is
 * [num_blocks][block_size = 16][n_kv_heads][head_dim] bf16, row-major. The
 * block table is int32 [n_seqs][max_blocks_per_seq]; logical position pos of
 * sequence b lives in slot block_table[b][pos / 16] * 16 + pos % 16.
 *
 * Attention (per sequence b, query head h, query at absolute position p):
 *   g    = h / (n_q_heads / n_kv_heads)                     GQA group
 *   J    = { j : j <= p and (window == 0 or p - j < window) }
 *   s_j  = scale * <q, K_j>;  s_j = softcap * tanh(s_j / softcap) if softcap > 0
 *   out  = sum_j softmax(s)_j V_j;   lse = log sum_j exp(s_j)  (natural log)
 * with V_j = K_j when k_eq_v (V aliases the K pages). The window rule is the
 * band rule of InfiniLM PR 581 ("feat: support gemma2 and gemma3_text",
 * Gemma-3 item 3): key j is hidden from chunk row i when past + i - j >= W,
 * composed with the aligned causal rule; decode is the row p = seq_len - 1,
 * which reads only the last min(seq_len, W) keys. The softcap sits on the
 * scaled score before mask and softmax (same PR, Gemma-2 item 1 and the
 * softcap section). Scale 1.0 is Gemma 4's (QK-norm; "MNN supports the full
 * Gemma4 family", section 6.1), 1/sqrt(query_pre_attn_scalar) is Gemma 2's.
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must be device memory of the current
 *    device (or managed memory); the library never copies host buffers.
 *    Every bf16 tensor pointer (q, k, v, pools) and every `out` must be
 *    16-byte aligned.
 *  - The caller owns every buffer: inputs, pools, tables, outputs and the
 *    workspace. The library allocates and frees nothing.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream) and do
 *    not synchronise the host, so they can be captured in CUDA graphs.
 *  - Return value: PSW_OK, or a negative PSW_E* code. Argument errors are
 *    detected on the host before anything is launched; nothing is written
 *    then. Errors that only the device can see (a block id outside
 *    [0, num_blocks), a sequence longer than its block-table row, a negative
 *    length) set bits in a per-device error word read by psw_get_error();
 *    the kernels skip the offending access and never trap.
 *  - Requires an sm_103 GPU (GB300); other devices return PSW_EDEVICE.
 */
#ifndef PSW_H
#define PSW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PSW_API __attribute__((visibility("default")))
#else
#define PSW_API
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *psw_stream_t;

/* ---- return codes (host-detected) ---- */
#define PSW_OK                 0
#define PSW_ENULL             -1  /* a required pointer is NULL */
#define PSW_EINVAL_HEADS      -2  /* n_q_heads or n_kv_heads <= 0, or n_q % n_kv != 0 */
#define PSW_EINVAL_HDIM       -3  /* head_dim not 256 or 512 */
#define PSW_EINVAL_SOFTCAP    -4  /* softcap negative or not finite */
#define PSW_EINVAL_WINDOW     -5  /* window negative */
#define PSW_EINVAL_BLOCKSIZE  -6  /* block_size != 16 */
#define PSW_EINVAL_KEQV       -7  /* k_eq_v with a V pointer, or V pointer missing */
#define PSW_EINVAL_SCALE      -8  /* scale <= 0 or not finite */
#define PSW_EINVAL_NSEQS      -9  /* n_seqs negative */
#define PSW_EWORKSPACE       -10  /* workspace smaller than psw_workspace_bytes() */
#define PSW_ECAPACITY        -11  /* max_blocks_per_seq or num_blocks <= 0, or
                                     max_seq_len > max_blocks_per_seq * 16 */
#define PSW_EALIGN           -12  /* a tensor pointer (bf16 inputs, pools, out) is not 16-byte aligned */
#define PSW_EDEVICE          -13  /* no usable sm_103 device */
#define PSW_ELAUNCH          -14  /* a CUDA launch or attribute call failed */
#define PSW_ETENSORMAP       -15  /* the TMA descriptor for a pool could not be built */
#define PSW_ESCRATCH         -16  /* the batch needs more scratch than the static buffer of
                                     attn_decode_paged_noalloc holds */
#define PSW_EINVAL_ROPE      -17  /* theta <= 0, partial_rotary_factor outside (0, 1], eps < 0,
                                     or one of them not finite */
#define PSW_EINVAL_LAYERS    -18  /* n_layers or pattern <= 0, n_shared outside [0, n_layers),
                                     or a shared layer with no cache-owning layer of its type */
#define PSW_ENOBLOCKS        -19  /* the block pool has fewer free blocks than asked for */
#define PSW_EBLOCK           -20  /* a block id outside the pool, or freed more often than held */

/* ---- device error bits (psw_get_error) ---- */
#define PSW_DEVERR_BLOCK_ID    1  /* block id outside [0, num_blocks): access skipped */
#define PSW_DEVERR_CAPACITY    2  /* sequence longer than its block-table row: clamped */
#define PSW_DEVERR_LENGTH      4  /* negative length or non-monotone offsets: row skipped */
#define PSW_DEVERR_PIPELINE    8  /* a bounded pipeline wait timed out: tile abandoned */

/* Per-layer attention parameters. */
typedef struct {
  int32_t n_q_heads;   /* query heads; n_q_heads % n_kv_heads == 0 */
  int32_t n_kv_heads;  /* key/value heads of this layer (may differ per layer) */
  int32_t head_dim;    /* 256 (sliding layers) or 512 (full layers) */
  int32_t window;      /* 0 = full causal attention; W > 0 = sliding window of W keys */
  float   softcap;     /* 0 = off; > 0 applies cap * tanh(s / cap) */
  float   scale;       /* multiplies q.k before the softcap; > 0 */
  int32_t k_eq_v;      /* 1: V reads the K pages and every V pointer must be NULL */
  int32_t block_size;  /* tokens per page; must be 16 */
} psw_layer_t;

/* Page table of one layer (device pointer, shared by all calls of a step). */
typedef struct {
  const int32_t *block_table;  /* device int32 [n_seqs][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;  /* row length of block_table */
  int64_t num_blocks;          /* blocks in each pool; valid ids are [0, num_blocks) */
} psw_pages_t;

/*
 * Workspace bytes that attn_decode_paged and attn_prefill_chunked need for a
 * batch of up to n_seqs sequences (max_seq_len bounds every seq_len and every
 * past_len + chunk length). Pure host arithmetic; needs no GPU. The same
 * workspace may be reused by consecutive calls on one stream; when several
 * calls share it, size it for the largest of them.
 *
 * Zeroing rule: the first PSW_WORKSPACE_COUNTER_BYTES bytes of a workspace
 * hold the merge tickets of attn_decode_paged. They must be zero before the
 * first call that uses the workspace (zero-fill the buffer once when it is
 * allocated); every call leaves them zero again, so no call needs a reset.
 * Only a call that flagged PSW_DEVERR_PIPELINE may leave them non-zero; zero
 * them again before reusing that workspace.
 * Returns PSW_OK and writes *bytes, or an argument error.
 */
#define PSW_WORKSPACE_COUNTER_BYTES 2048
PSW_API int psw_workspace_bytes(const psw_layer_t *layer, int32_t n_seqs, int32_t max_seq_len,
                        size_t *bytes);

/*
 * reshape_and_cache ("Gemma 4 model architecture analysis", section 6.4):
 * token t of sequence b (cu_new[b] <= t < cu_new[b+1]) has logical position
 * past_lens[b] + (t - cu_new[b]); its K row k[t] (n_kv_heads x head_dim bf16)
 * is copied bit for bit into that position's slot of k_pool, and v[t] into
 * v_pool. With k_eq_v, v and v_pool must be NULL and only K is written.
 *   k, v       device bf16 [n_new_total][n_kv_heads][head_dim], n_new_total = cu_new[n_seqs]
 *   cu_new     device int32 [n_seqs + 1], non-decreasing, cu_new[0] = 0
 *   past_lens  device int32 [n_seqs], tokens already cached per sequence
 *   pages      block table of the pools; it must cover every written position
 *   k_pool, v_pool  device bf16 [num_blocks][16][n_kv_heads][head_dim], written
 * Slots whose block id falls outside the pool are skipped and flagged
 * (PSW_DEVERR_BLOCK_ID); every other slot of the pools is left untouched.
 */
PSW_API int kv_cache_write(const psw_layer_t *layer, const void *k, const void *v,
                   const int32_t *cu_new, const int32_t *past_lens, int32_t n_seqs,
                   const psw_pages_t *pages, void *k_pool, void *v_pool,
                   psw_stream_t stream);

/*
 * Decode attention: sequence b has seq_lens[b] cached tokens, the last of
 * which is the query's own (write it with kv_cache_write first); its single
 * query q[b] sits at position seq_lens[b] - 1. Sliding layers read only the
 * last min(seq_len, window) keys.
 *   q          device bf16 [n_seqs][n_q_heads][head_dim]
 *   k_pool     device bf16 pool; v_pool likewise, NULL when k_eq_v
 *   seq_lens   device int32 [n_seqs]; 0 gives a zero row and lse = -inf
 *   out        device fp32 [n_seqs][n_q_heads][head_dim]
 *   lse        device fp32 [n_seqs][n_q_heads] or NULL
 *   ws         device workspace of ws_bytes >= psw_workspace_bytes(layer, n_seqs, .),
 *              zero-filled once before its first use (see the zeroing rule above)
 * Split-KV flash decoding in one kernel launch: every CTA derives its share of
 * the work from seq_lens, partial results over page ranges go to the
 * workspace, and the CTA that finishes a sequence's last range combines them
 * with the log-sum-exp rule.
 */
PSW_API int attn_decode_paged(const psw_layer_t *layer, const void *q, const void *k_pool,
                      const void *v_pool, const psw_pages_t *pages,
                      const int32_t *seq_lens, int32_t n_seqs, float *out, float *lse,
                      void *ws, size_t ws_bytes, psw_stream_t stream);

/*
 * One decode step in one launch: kv_cache_write of each sequence's new token
 * followed by attn_decode_paged, fused. Sequence b's new K/V row (the query's
 * own token, position seq_lens[b] - 1) is stored in its slot of the pools and
 * attended to in the same pass: the kernel that stages the page holding it
 * takes the row from k_new / v_new instead of the pool, so no second launch
 * and no ordering between the two is needed. Results and pools equal those of
 * kv_cache_write (cu_new = 0..n_seqs, past_lens = seq_lens - 1) then
 * attn_decode_paged.
 *   k_new, v_new  device bf16 [n_seqs][n_kv_heads][head_dim], 16-byte aligned;
 *                 v_new NULL when k_eq_v
 *   k_pool, v_pool  as attn_decode_paged, written at the new slots
 * Every other argument, the workspace and the errors are those of
 * attn_decode_paged (PSW_ENULL for a missing k_new; PSW_EINVAL_KEQV when
 * v_new breaks the k_eq_v rule). A sequence of length 0 writes nothing; a
 * new slot with a bad block id or beyond the table row is skipped and flagged
 * as by kv_cache_write.
 */
PSW_API int attn_decode_paged_append(const psw_layer_t *layer, const void *q, const void *k_new,
                                     const void *v_new, void *k_pool, void *v_pool,
                                     const psw_pages_t *pages, const int32_t *seq_lens,
                                     int32_t n_seqs, float *out, float *lse, void *ws,
                                     size_t ws_bytes, psw_stream_t stream);

/*
 * Chunked prefill: sequence b contributes the chunk rows
 * cu_q[b] <= t < cu_q[b+1]; row i = t - cu_q[b] sits at position
 * past_lens[b] + i and attends over keys [0, past_lens[b] + i] under the band
 * and causal rules. The chunk's own K/V must already be in the pages
 * (kv_cache_write first).
 *   q          device bf16 [n_q_total][n_q_heads][head_dim]
 *   cu_q       device int32 [n_seqs + 1], non-decreasing, cu_q[n_seqs] <= n_q_total
 *   past_lens  device int32 [n_seqs]
 *   n_q_total  host: rows of q and out
 *   max_q_len  host bound on every chunk length (cu_q[b+1] - cu_q[b]); longer
 *              chunks are flagged (PSW_DEVERR_LENGTH) and their excess rows skipped
 *   out        device fp32 [n_q_total][n_q_heads][head_dim]; lse fp32 [n_q_total][n_q_heads] or NULL
 *   ws         device workspace of ws_bytes >= psw_workspace_bytes(layer, n_seqs, L)
 *              for any L >= max_q_len; it holds the work list of the call after
 *              the counter block, which this call neither reads nor writes
 * Tensor-core kernel (tcgen05 MMAs with S, P and O in tensor memory, K/V tiles
 * fed by TMA through the block table); key tiles that the band rule hides from
 * every row of a query tile are never loaded. A small plan kernel first orders
 * the work (blocks of 128 / G chunk tokens per KV head) longest first; a
 * persistent grid then takes it in that order. Needs n_q_heads / n_kv_heads
 * <= 128 and n_seqs <= 65535; PSW_EWORKSPACE when ws is missing or too small.
 */
PSW_API int attn_prefill_chunked(const psw_layer_t *layer, const void *q, const int32_t *cu_q,
                         const int32_t *past_lens, int32_t n_seqs, int32_t n_q_total,
                         int32_t max_q_len,
                         const void *k_pool, const void *v_pool, const psw_pages_t *pages,
                         float *out, float *lse, void *ws, size_t ws_bytes,
                         psw_stream_t stream);

/*
 * attn_decode_paged for callers that cannot allocate device memory (their
 * device memory belongs to another allocator with a fixed budget, or they must
 * not call cudaMalloc once serving has started). The pages have no counterpart
 * for this entry point; it is a property of this library only.
 *
 * Arguments, results and errors are those of attn_decode_paged, without the
 * workspace: the scratch comes from a static device buffer of
 * PSW_NOALLOC_SCRATCH_BYTES inside the library. Pointer and alignment errors
 * are reported first, as by attn_decode_paged; then a batch whose workspace
 * (psw_workspace_bytes) exceeds the buffer returns PSW_ESCRATCH before
 * anything runs: with head_dim 256 that is more than about 1500 units, with
 * head_dim 512 more than about 500, where units = n_seqs * n_kv_heads *
 * ceil((n_q_heads / n_kv_heads) / 8).
 *
 * Set-up: the first call on a device looks up the buffer's device address
 * (with that device current) and keeps it. Under CUDA's lazy module loading
 * (the default) that lookup is also when the driver loads the library's
 * module holding the buffer and reserves its memory on the device, so that
 * step can fail (PSW_EDEVICE) if the device is out of memory. Make the first
 * call at start-up, before any stream capture: a call with n_seqs = 0 and
 * valid pointers does the set-up and launches nothing. From then on the
 * buffer stays reserved on that device until the process exits, and nothing
 * is allocated or freed by this entry point.
 *
 * All calls share the buffer and it keeps the last call's contents; its
 * counters start at zero (static storage) and every call leaves them zero.
 * Calls whose kernels could overlap on the GPU (several streams or host
 * threads on one device) race on the buffer: serialise them.
 */
#define PSW_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)
PSW_API int attn_decode_paged_noalloc(const psw_layer_t *layer, const void *q,
                                      const void *k_pool, const void *v_pool,
                                      const psw_pages_t *pages, const int32_t *seq_lens,
                                      int32_t n_seqs, float *out, float *lse,
                                      psw_stream_t stream);

/* Parameters of the pre-attention step of one layer. */
typedef struct {
  float theta;                  /* RoPE base: 10000 on sliding layers, 1e6 on full layers */
  float partial_rotary_factor;  /* fraction of head_dim that is rotated, in (0, 1] */
  float eps;                    /* RMS-norm epsilon, >= 0 */
  const float *q_weight;        /* device fp32 [head_dim]: effective q_norm weight, or NULL */
  const float *k_weight;        /* device fp32 [head_dim]: effective k_norm weight, or NULL */
  const float *v_weight;        /* device fp32 [head_dim]: v_norm weight, or NULL (weightless) */
} psw_norm_rope_t;

/*
 * The step before attention, fused into one kernel: per-head RMS-norm of the
 * new tokens' q, k and v, the proportional rotary embedding of q and k, and
 * the cache write of k and v.
 *
 * Per head vector x (head_dim elements) of token t of sequence b, at position
 * pos = past_lens[b] + (t - cu_new[b]):
 *   y_d = x_d / sqrt(mean(x^2) + eps) * w_d        (w_d = 1 without a weight)
 * (RMS-norm per head vector before the rotation: InfiniLM PR 581, Gemma-3
 * item 1, whose weights are stored as w - 1 and loaded as w: pass the loaded
 * weight; v_norm: "MNN supports the full Gemma4 family", section 6.1). For q
 * and k only (V is not rotated, same page section 6.2), the proportional
 * rotary embedding of "Gemma 4 model architecture analysis", challenge 5:
 * with rope_angles = floor(partial_rotary_factor * head_dim / 2), pair i of
 * dims (i, i + head_dim / 2) turns by a = pos * theta^(-2 i / head_dim) for
 * i < rope_angles (the head size, not the rotated size, is the exponent's
 * denominator) and not at all beyond:
 *   out_i = y_i cos a - y_{i + hd/2} sin a,  out_{i + hd/2} = y_{i + hd/2} cos a + y_i sin a.
 * The rotate-half pairing is this library's reading; the pages do not print
 * the pairing. Results are rounded to bf16 (nearest, ties to even):
 *   q_out  device bf16 [n_new_total][n_q_heads][head_dim]; may be q itself
 *   k_pool, v_pool  receive the rotated k and the normalised v rows in the
 *          slot block_table[b][pos / 16] * 16 + pos % 16, as kv_cache_write
 * Inputs: q device bf16 [n_new_total][n_q_heads][head_dim]; k, v device bf16
 * [n_new_total][n_kv_heads][head_dim]; cu_new, past_lens as kv_cache_write.
 * A layer whose V aliases its K pages (k_eq_v) passes v = v_pool = NULL. A
 * Gemma-4 layer whose V comes from the K projection (different from K: only
 * normalised) is a k_eq_v = 0 layer that passes the same raw k buffer as v.
 * A layer that reads another layer's cache (KV sharing) passes k = v =
 * k_pool = v_pool = NULL (and may pass pages = NULL): only q is processed.
 * Errors: those of kv_cache_write, PSW_EINVAL_ROPE and PSW_ENULL for a
 * missing rn, q or q_out (any number of heads per token is accepted: the
 * kernel takes a token's head vectors eight at a time, four at head_dim
 * 512). Device-side errors are flagged
 * as by kv_cache_write: a token whose block id or capacity is wrong still
 * gets its q_out rows (only its K/V write is skipped); a token with an
 * invalid length or offsets is skipped.
 */
PSW_API int qkv_norm_rope_cache_write(const psw_layer_t *layer, const psw_norm_rope_t *rn,
                                      const void *q, const void *k, const void *v,
                                      const int32_t *cu_new, const int32_t *past_lens,
                                      int32_t n_seqs, const psw_pages_t *pages, void *q_out,
                                      void *k_pool, void *v_pool, psw_stream_t stream);

/*
 * ---- FP8 KV pages (e4m3), halving the bytes decode reads
 *
 * The pages name no KV quantisation (InfiniLM PR 581's hardening table
 * refuses it for sliding layers); this is the library's own format. A pool
 * holds one-byte OCP E4M3 codes in the bf16 pool's layout,
 * uint8 [num_blocks][16][n_kv_heads][head_dim], with a scale pool fp32
 * [num_blocks][16][n_kv_heads]: one scale per (slot, KV head) row, so the
 * tokens of a page can be written one at a time. For a row x:
 *   scale = amax / 448, code_d = e4m3(x_d * (448 / amax)), amax = max |x|
 * (fp32 division and product rounded to nearest; the conversion rounds to
 * nearest even and saturates at 448; an all-zero row has scale 0). The row
 * stands for code_d * scale; attention runs on those values exactly (codes
 * convert to bf16 without loss, the K scale multiplies the score, the V
 * scale multiplies P).
 */

/* kv_cache_write into FP8 pools: arguments as kv_cache_write, with
 * k_pool8 / v_pool8 the code pools and k_scale / v_scale (device fp32,
 * 4-byte aligned) the scale pools; with k_eq_v, v, v_pool8 and v_scale are
 * NULL. Errors as kv_cache_write. */
PSW_API int kv_cache_write_fp8(const psw_layer_t *layer, const void *k, const void *v,
                               const int32_t *cu_new, const int32_t *past_lens,
                               int32_t n_seqs, const psw_pages_t *pages, void *k_pool8,
                               void *v_pool8, float *k_scale, float *v_scale,
                               psw_stream_t stream);

/* attn_decode_paged over FP8 pools (arguments, results, workspace and errors
 * as attn_decode_paged; v_pool8 and v_scale NULL with k_eq_v). The same
 * split-KV kernel streams e4m3 tiles (half the bytes) and converts them to
 * bf16 in shared memory before its matrix products. */
PSW_API int attn_decode_paged_fp8(const psw_layer_t *layer, const void *q, const void *k_pool8,
                                  const void *v_pool8, const float *k_scale,
                                  const float *v_scale, const psw_pages_t *pages,
                                  const int32_t *seq_lens, int32_t n_seqs, float *out,
                                  float *lse, void *ws, size_t ws_bytes, psw_stream_t stream);

/*
 * Layer types of a hybrid stack and its KV-sharing map. Host arithmetic only
 * (no GPU, nothing launched).
 *   is_full[i] = 1 when (i + 1) % pattern == 0, else 0 (sliding): the
 *     interleaving rule of InfiniLM PR 581, Gemma-3 item 2 (pattern 6 gives
 *     Gemma-3's 5:1 stack).
 *   target[i]  = i for the first n_layers - n_shared layers, which own their
 *     caches; each of the last n_shared layers reads the cache of the last
 *     cache-owning layer of its own type and writes none ("MNN supports the
 *     full Gemma4 family", KV-sharing section: in the 35-layer E2B with
 *     pattern 5 and 20 shared layers, sliding layers read layer 13 and full
 *     layers read layer 14; "Gemma 4 model architecture analysis", section 4:
 *     a shared layer keeps its own q projection, skips the cache write and
 *     attends over its target's pages).
 * A shared layer runs qkv_norm_rope_cache_write with k = v = NULL and then
 * the attention calls on its target's pools and block table.
 * Either output pointer may be NULL. Returns PSW_OK or PSW_EINVAL_LAYERS.
 */
PSW_API int psw_kv_share_map(int32_t n_layers, int32_t pattern, int32_t n_shared,
                             int32_t *is_full, int32_t *target);

/*
 * ---- host page allocator with prefix caching (no GPU involved)
 *
 * The abstractions of "Gemma 4 model architecture analysis" (vLLM-Kunlun),
 * section 6.2: each physical page (block) carries {block_id, ref_cnt,
 * block_hash}; the pool keeps unreferenced pages in a free queue in
 * least-recently-freed order; a sequence's block-table row lists its pages
 * (the int32 rows every attention call takes). Section 6.6, prefix caching:
 * a full page is named by the hash of its 16 tokens chained with the previous
 * page's hash, and a request whose prefix matches cached pages shares those
 * physical pages (a hit raises the page's reference count; the KV of those
 * tokens is not computed again). Freed pages keep their hash until the queue
 * hands them out again, so a later request can still hit them.
 * The hash is FNV-1a over 64 bits (the parent hash as 8 little-endian bytes,
 * then each token as 4): not a cryptographic hash; two different prefixes
 * collide with probability about n^2 / 2^65 for n cached pages.
 * Every call takes the pool's lock. Block ids are int32 in [0, num_blocks).
 */
typedef struct psw_block_pool psw_block_pool_t;

/* Creates a pool of num_blocks free pages (prefix caching on when
 * enable_prefix_cache != 0). PSW_ECAPACITY for num_blocks outside
 * [1, 2^31 - 1], PSW_ENOBLOCKS when the host allocation fails. */
PSW_API int psw_block_pool_create(int64_t num_blocks, int32_t enable_prefix_cache,
                                  psw_block_pool_t **pool_out);
PSW_API void psw_block_pool_destroy(psw_block_pool_t *pool);
/* Pages with ref_cnt 0 (in the free queue), or PSW_ENULL. */
PSW_API int64_t psw_block_pool_num_free(psw_block_pool_t *pool);
/* Takes n pages from the head of the free queue (least recently freed
 * first), each with ref_cnt 1; a page that still carried a hash loses it.
 * All or nothing: PSW_ENOBLOCKS when fewer than n are free. */
PSW_API int psw_block_pool_allocate(psw_block_pool_t *pool, int32_t n, int32_t *ids_out);
/* ref_cnt -= 1 for each id, in order; a page reaching 0 joins the tail of
 * the free queue and keeps its hash. PSW_EBLOCK (nothing changed) for an id
 * outside the pool or released more often than it is held. Freeing a
 * sequence's row back to front puts its last pages first in line for reuse. */
PSW_API int psw_block_pool_free(psw_block_pool_t *pool, const int32_t *ids, int32_t n);
/* get_cached_block: the page cached under `hash` gets ref_cnt += 1 (leaving
 * the free queue if it was there) and its id is returned; -1 on a miss. */
PSW_API int psw_block_pool_get_cached(psw_block_pool_t *pool, uint64_t hash, int32_t *id_out);
/* Names a referenced page by the hash of its (now written) tokens; a hash
 * already naming another page keeps that page. PSW_EBLOCK for a page not
 * held by anyone. */
PSW_API int psw_block_pool_cache(psw_block_pool_t *pool, int32_t id, uint64_t hash);
PSW_API int psw_block_pool_ref_count(psw_block_pool_t *pool, int32_t id, int32_t *ref_out);
/* Chained page hash: FNV-1a of (parent, tokens[0..n)). The first page's
 * parent is 0. */
PSW_API uint64_t psw_block_hash(uint64_t parent, const int32_t *tokens, int32_t n);
/* Admits a request of n_tokens prompt tokens: walks its full pages (all but
 * the page holding the last token, whose query must run) through the prefix
 * cache until the first miss, then allocates the rest. Writes the block-table
 * row (ceil(n_tokens / 16) ids, -1 up to max_blocks) and the number of
 * leading tokens whose KV is already in the pages (the request's past length
 * for its first prefill chunk). On an error nothing stays held. */
PSW_API int psw_block_pool_admit(psw_block_pool_t *pool, const int32_t *tokens,
                                 int32_t n_tokens, int32_t *table_row, int32_t max_blocks,
                                 int32_t *n_cached_tokens);
/* After the request's KV is written: names each full page of the row by its
 * chained hash so that later requests can share it. */
PSW_API int psw_block_pool_commit(psw_block_pool_t *pool, const int32_t *tokens,
                                  int32_t n_tokens, const int32_t *table_row);

/*
 * Synchronises `stream`, then returns the current device's error word (an OR
 * of PSW_DEVERR_* bits, 0 when nothing was flagged) in *device_error_out and
 * clears it. Returns PSW_OK or PSW_ELAUNCH when the stream reports an error.
 */
PSW_API int psw_get_error(psw_stream_t stream, int32_t *device_error_out);

/* Static string describing a return code. */
PSW_API const char *psw_strerror(int code);

/*
 * Testing hook for the bounded pipeline waits; not for production use.
 * kernel 1 (attn_decode_paged, attn_decode_paged_fp8) or 2
 * (attn_prefill_chunked): from the next launch of that kernel on, the TMA
 * producer of CTA `cta` leaves its copy number `tile` (counted from 0 over its
 * own K-tile copies) unissued and stops, without flagging anything. The
 * consumer waiting for that copy then gives up after its bound (about one
 * second), sets PSW_DEVERR_PIPELINE and abandons the CTA's remaining work;
 * the producer still waits for every copy it did issue, and the prefill
 * kernel still frees its tensor memory, before the CTA exits. Outputs of the
 * abandoned work are left unwritten, and a decode call may leave the
 * workspace's counter block non-zero (zero it before the next call). kernel 0
 * switches the hook off. Returns PSW_OK, or PSW_EINVAL_NSEQS for a kernel
 * outside [0, 2] or a negative cta or tile.
 */
PSW_API int psw_testing_stall(int32_t kernel, int32_t cta, int32_t tile);

#ifdef __cplusplus
}
#endif

#endif /* PSW_H */
