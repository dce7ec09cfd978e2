/*
 * psw_oracle.c -- plain fp64 CPU oracle for paged sliding-window attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file. It shares no code, header, table or helper
 * with the CUDA library; the two meet only through the seeded inputs.
 *
 * What it computes, and where the pages define it:
 *
 *  - Slot mapping: slot = block_table[r][pos / bs] * bs + pos % bs
 *    ("Gemma 4 model architecture analysis" (vLLM-Kunlun), section 6.3,
 *    key formula and its worked example; the block table is the page table of
 *    section 6.2).
 *  - Cache write (reshape_and_cache): every new token's K row and V row is
 *    copied to key_cache[block_id, offset, :, :] and value_cache[...], a pool
 *    laid out [num_blocks, block_size, n_kv_heads, head_dim] (same page,
 *    section 6.4).
 *  - Attention for one query at absolute position p of sequence b (the paged
 *    read of section 6.5; masking and softcap from InfiniLM PR 581
 *    "feat: support gemma2 and gemma3_text", Gemma-2 item 1 and Gemma-3
 *    item 3; scale 1.0 from "MNN supports the full Gemma4 family", section
 *    6.1; GQA grouping from "Gemma 4 architecture decoded", GQA section):
 *        g   = h / (n_q / n_kv)                    (contiguous GQA groups)
 *        J   = { j : 0 <= j <= p  and  (W == 0 or p - j < W) }
 *        s_j = scale * sum_d q_d K_{j,d}
 *        s_j = cap * tanh(s_j / cap)                (only when cap > 0)
 *        out = sum_j softmax(s)_j V_j,  lse = log sum_j exp(s_j)
 *    with V_j = K_j when k_eq_v is set (V aliases the K pages).
 *    Decode uses p = seq_len - 1 (only the last min(seq_len, W) keys are
 *    visible); chunked prefill uses p = past + i for chunk row i, which is the
 *    band rule "key j hidden from query i when past + i - j >= W" composed
 *    with the aligned causal rule.
 *  - KV-cache size: batch * seq * layers * n_kv * head_dim * bytes, doubled
 *    when a separate V cache is kept (the KV-size worked example in
 *    "Gemma 4 architecture decoded", GQA section).
 *  - The pre-attention step: per-head RMS-norm of q, k and v, then the
 *    proportional rotary embedding of q and k (see oracle_norm_rope_row).
 *
 * Arithmetic: bf16 inputs are widened exactly to double; every sum, the
 * softcap, the exponentials and the normalisation run in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Physical slot of logical position `pos` for one block-table row. */
int64_t oracle_slot(const int32_t *block_table_row, int64_t pos, int32_t block_size)
{
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    return (int64_t)block_table_row[logical_block] * block_size + offset;
}

/* Bytes of KV cache for the given shape; with_v = 0 counts K only. */
double oracle_kv_cache_bytes(int64_t batch, int64_t seq_len, int64_t n_layers,
                             int64_t n_kv_heads, int64_t head_dim,
                             int64_t dtype_bytes, int32_t with_v)
{
    double one = (double)batch * (double)seq_len * (double)n_layers *
                 (double)n_kv_heads * (double)head_dim * (double)dtype_bytes;
    return with_v ? 2.0 * one : one;
}

/*
 * reshape_and_cache: token t of sequence b (t counted from cu_new[b]) sits at
 * logical position past_lens[b] + (t - cu_new[b]). v_pool may be NULL, in
 * which case no V row is written (V aliases the K pages).
 * Returns 0, or -1 when a block id falls outside [0, num_blocks) (nothing is
 * written for that row).
 */
int32_t oracle_kv_cache_write(const uint16_t *k_new, const uint16_t *v_new,
                              const int32_t *cu_new, const int32_t *past_lens,
                              int32_t n_seqs, const int32_t *block_table,
                              int32_t max_blocks_per_seq, int64_t num_blocks,
                              int32_t n_kv_heads, int32_t head_dim,
                              int32_t block_size, uint16_t *k_pool,
                              uint16_t *v_pool)
{
    int32_t status = 0;
    int64_t row_elems = (int64_t)n_kv_heads * head_dim;
    for (int32_t b = 0; b < n_seqs; ++b) {
        const int32_t *row = block_table + (int64_t)b * max_blocks_per_seq;
        for (int32_t t = cu_new[b]; t < cu_new[b + 1]; ++t) {
            int64_t pos = (int64_t)past_lens[b] + (t - cu_new[b]);
            int64_t slot = oracle_slot(row, pos, block_size);
            int64_t block_id = slot / block_size;
            if (block_id < 0 || block_id >= num_blocks) {
                status = -1;
                continue;
            }
            memcpy(k_pool + slot * row_elems, k_new + (int64_t)t * row_elems,
                   (size_t)row_elems * sizeof(uint16_t));
            if (v_pool != NULL)
                memcpy(v_pool + slot * row_elems, v_new + (int64_t)t * row_elems,
                       (size_t)row_elems * sizeof(uint16_t));
        }
    }
    return status;
}

typedef struct {
    /* layer */
    int32_t n_q_heads, n_kv_heads, head_dim, window, block_size, k_eq_v;
    double softcap, scale;
    /* inputs */
    const uint16_t *q_rows;   /* [n_rows, n_q_heads, head_dim] */
    const int32_t *row_seq;   /* [n_rows] */
    const int64_t *row_pos;   /* [n_rows]; < 0 means an empty row */
    int64_t n_rows;
    const uint16_t *k_pool, *v_pool;
    /* FP8 pages (fp8 != 0): e4m3 codes and one scale per (slot, KV head) */
    int32_t fp8;
    const uint8_t *k8, *v8;
    const float *k_scale, *v_scale;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    /* outputs */
    double *out;              /* [n_rows, n_q_heads, head_dim] */
    double *lse;              /* [n_rows, n_q_heads] */
    /* work split */
    int32_t n_threads;
    int32_t thread_index;
} attn_job_t;

/*
 * ---- FP8 KV pages (e4m3 codes, one fp32 scale per slot and KV head)
 *
 * The pages name no KV quantisation (InfiniLM PR 581's hardening table
 * refuses it for sliding layers); this library's format is the OCP FP8
 * E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448; subnormals m * 2^-9)
 * with a per-row scale: for a row x of head_dim values with amax = max |x|,
 *   scale = amax / 448 and code_d = e4m3(x_d * (448 / amax)),
 * both fp32 operations rounded to nearest, the conversion rounding to
 * nearest even and saturating at 448; an all-zero row has scale 0 and codes
 * 0. The value a code stands for is code * scale (exact in double).
 */
double oracle_e4m3_decode(uint8_t c)
{
    int neg = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return neg ? -v : v;
}

uint8_t oracle_e4m3_encode(float x)
{
    if (x != x)
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E; /* saturate to the largest finite value */
    int e;
    (void)frexp(a, &e); /* a = f * 2^e, 0.5 <= f < 1: a in [2^(e-1), 2^e) */
    int q = e - 1 - 3;  /* quantum of a normal code in that binade */
    if (q < -9)
        q = -9; /* subnormal quantum */
    double n = nearbyint(ldexp(a, -q)); /* ties to even */
    double v = ldexp(n, q);
    if (v == 0.0)
        return sign;
    if (v >= 448.0)
        return sign | 0x7E;
    if (v < 0.015625) /* below 2^-6: subnormal code m * 2^-9 */
        return sign | (uint8_t)n;
    int ev;
    double f = frexp(v, &ev); /* v = f * 2^ev, f in [0.5, 1) */
    int mant = (int)((f * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(((ev - 1 + 7) << 3) | mant);
}

/* One row of the per-row quantisation (see above). */
static void quantize_row(const uint16_t *x, int32_t n, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int32_t d = 0; d < n; ++d) {
        uint32_t u = ((uint32_t)x[d]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        if (fabsf(f) > amax)
            amax = fabsf(f);
    }
    if (amax == 0.0f) {
        *scale = 0.0f;
        memset(codes, 0, (size_t)n);
        return;
    }
    float inv = 448.0f / amax;
    *scale = amax / 448.0f;
    for (int32_t d = 0; d < n; ++d) {
        uint32_t u = ((uint32_t)x[d]) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        codes[d] = oracle_e4m3_encode(f * inv);
    }
}

/*
 * reshape_and_cache into FP8 pages: as oracle_kv_cache_write, but each
 * (token, KV head) row of head_dim values is quantised into its slot's codes
 * (pools uint8 [num_blocks][block_size][n_kv][head_dim]) and scale (fp32
 * [num_blocks][block_size][n_kv]). v8 / v_scale NULL: K only.
 */
int32_t oracle_kv_cache_write_fp8(const uint16_t *k_new, const uint16_t *v_new,
                                  const int32_t *cu_new, const int32_t *past_lens,
                                  int32_t n_seqs, const int32_t *block_table,
                                  int32_t max_blocks_per_seq, int64_t num_blocks,
                                  int32_t n_kv_heads, int32_t head_dim,
                                  int32_t block_size, uint8_t *k8, uint8_t *v8,
                                  float *k_scale, float *v_scale)
{
    int32_t status = 0;
    for (int32_t b = 0; b < n_seqs; ++b) {
        const int32_t *row = block_table + (int64_t)b * max_blocks_per_seq;
        for (int32_t t = cu_new[b]; t < cu_new[b + 1]; ++t) {
            int64_t pos = (int64_t)past_lens[b] + (t - cu_new[b]);
            int64_t slot = oracle_slot(row, pos, block_size);
            int64_t block_id = slot / block_size;
            if (block_id < 0 || block_id >= num_blocks) {
                status = -1;
                continue;
            }
            for (int32_t g = 0; g < n_kv_heads; ++g) {
                int64_t src = ((int64_t)t * n_kv_heads + g) * head_dim;
                int64_t dst = slot * n_kv_heads + g;
                quantize_row(k_new + src, head_dim, k8 + dst * head_dim, &k_scale[dst]);
                if (v8 != NULL)
                    quantize_row(v_new + src, head_dim, v8 + dst * head_dim, &v_scale[dst]);
            }
        }
    }
    return status;
}

/* Values of a K or V row (bf16 pages, or FP8 codes times their scale). */
static void kv_row(const attn_job_t *job, const uint16_t *pool16, const uint8_t *pool8,
                   const float *scale8, int64_t slot, int32_t g, double *out)
{
    const int32_t hd = job->head_dim;
    const int64_t r = slot * job->n_kv_heads + g;
    if (job->fp8) {
        const double s = (double)scale8[r];
        for (int32_t d = 0; d < hd; ++d)
            out[d] = oracle_e4m3_decode(pool8[r * hd + d]) * s;
    } else {
        for (int32_t d = 0; d < hd; ++d)
            out[d] = bf16_bits_to_double(pool16[r * hd + d]);
    }
}

static void attend_one(const attn_job_t *job, int64_t row, int32_t h,
                       double *scores, double *acc)
{
    const int32_t hd = job->head_dim;
    const int32_t group = job->n_q_heads / job->n_kv_heads;
    const int32_t g = h / group;
    const int64_t p = job->row_pos[row];
    const int32_t *bt_row =
        job->block_table + (int64_t)job->row_seq[row] * job->max_blocks_per_seq;
    const uint16_t *q = job->q_rows + (row * job->n_q_heads + h) * (int64_t)hd;
    const uint16_t *v_pool = job->k_eq_v ? job->k_pool : job->v_pool;
    const uint8_t *v8 = job->k_eq_v ? job->k8 : job->v8;
    const float *v_scale = job->k_eq_v ? job->k_scale : job->v_scale;
    double *out = job->out + (row * job->n_q_heads + h) * (int64_t)hd;
    double *kv = acc + hd; /* one K or V row */

    for (int32_t d = 0; d < hd; ++d)
        out[d] = 0.0;
    if (p < 0) { /* no keys at all: zero output, lse = -inf */
        job->lse[row * job->n_q_heads + h] = -INFINITY;
        return;
    }

    /* scores over every position 0..p, visibility decided per key */
    double m = -INFINITY;
    for (int64_t j = 0; j <= p; ++j) {
        int visible = (job->window == 0) || (p - j < job->window);
        if (!visible) {
            scores[j] = NAN; /* never read */
            continue;
        }
        int64_t slot = oracle_slot(bt_row, j, job->block_size);
        kv_row(job, job->k_pool, job->k8, job->k_scale, slot, g, kv);
        double dot = 0.0;
        for (int32_t d = 0; d < hd; ++d)
            dot += bf16_bits_to_double(q[d]) * kv[d];
        double s = job->scale * dot;
        if (job->softcap > 0.0)
            s = job->softcap * tanh(s / job->softcap);
        scores[j] = s;
        if (s > m)
            m = s;
    }

    double l = 0.0;
    for (int32_t d = 0; d < hd; ++d)
        acc[d] = 0.0;
    for (int64_t j = 0; j <= p; ++j) {
        int visible = (job->window == 0) || (p - j < job->window);
        if (!visible)
            continue;
        double w = exp(scores[j] - m);
        l += w;
        int64_t slot = oracle_slot(bt_row, j, job->block_size);
        kv_row(job, v_pool, v8, v_scale, slot, g, kv);
        for (int32_t d = 0; d < hd; ++d)
            acc[d] += w * kv[d];
    }
    for (int32_t d = 0; d < hd; ++d)
        out[d] = acc[d] / l;
    job->lse[row * job->n_q_heads + h] = m + log(l);
}

static void *attn_worker(void *arg)
{
    const attn_job_t *job = (const attn_job_t *)arg;
    int64_t max_pos = 0;
    for (int64_t r = 0; r < job->n_rows; ++r)
        if (job->row_pos[r] > max_pos)
            max_pos = job->row_pos[r];
    double *scores = (double *)malloc((size_t)(max_pos + 1) * sizeof(double));
    double *acc = (double *)malloc((size_t)job->head_dim * 2 * sizeof(double));
    if (scores == NULL || acc == NULL) {
        free(scores);
        free(acc);
        return (void *)1;
    }
    int64_t n_pairs = job->n_rows * job->n_q_heads;
    for (int64_t pair = job->thread_index; pair < n_pairs; pair += job->n_threads)
        attend_one(job, pair / job->n_q_heads, (int32_t)(pair % job->n_q_heads),
                   scores, acc);
    free(scores);
    free(acc);
    return NULL;
}

int32_t oracle_num_cores(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int32_t)n : 1;
}

/* Attention rows over bf16 pages or (fp8 != 0) FP8 pages. */
static int32_t attention_rows(int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t head_dim, int32_t window, double softcap,
                              double scale, int32_t k_eq_v, int32_t block_size,
                              const uint16_t *q_rows, const int32_t *row_seq,
                              const int64_t *row_pos, int64_t n_rows,
                              const uint16_t *k_pool, const uint16_t *v_pool,
                              int32_t fp8, const uint8_t *k8, const uint8_t *v8,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_table,
                              int32_t max_blocks_per_seq, double *out,
                              double *lse, int32_t n_threads)
{
    if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0 ||
        head_dim <= 0 || window < 0 || softcap < 0.0 || block_size <= 0)
        return -1;
    if (!fp8 && !k_eq_v && v_pool == NULL)
        return -1;
    if (fp8 && (k8 == NULL || k_scale == NULL || (!k_eq_v && (v8 == NULL || v_scale == NULL))))
        return -1;
    if (n_threads <= 0)
        n_threads = oracle_num_cores();
    if (n_rows * n_q_heads < n_threads)
        n_threads = (int32_t)(n_rows * n_q_heads > 0 ? n_rows * n_q_heads : 1);

    attn_job_t *jobs = (attn_job_t *)calloc((size_t)n_threads, sizeof(attn_job_t));
    pthread_t *threads = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (jobs == NULL || threads == NULL) {
        free(jobs);
        free(threads);
        return -2;
    }
    int32_t failed = 0;
    for (int32_t t = 0; t < n_threads; ++t) {
        attn_job_t *j = &jobs[t];
        j->n_q_heads = n_q_heads;
        j->n_kv_heads = n_kv_heads;
        j->head_dim = head_dim;
        j->window = window;
        j->block_size = block_size;
        j->k_eq_v = k_eq_v;
        j->softcap = softcap;
        j->scale = scale;
        j->q_rows = q_rows;
        j->row_seq = row_seq;
        j->row_pos = row_pos;
        j->n_rows = n_rows;
        j->k_pool = k_pool;
        j->v_pool = v_pool;
        j->fp8 = fp8;
        j->k8 = k8;
        j->v8 = v8;
        j->k_scale = k_scale;
        j->v_scale = v_scale;
        j->block_table = block_table;
        j->max_blocks_per_seq = max_blocks_per_seq;
        j->out = out;
        j->lse = lse;
        j->n_threads = n_threads;
        j->thread_index = t;
    }
    int32_t started = 0;
    for (int32_t t = 1; t < n_threads; ++t) {
        if (pthread_create(&threads[t], NULL, attn_worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* threads that failed to start are run inline */
    for (int32_t t = started + 1; t < n_threads; ++t)
        if (attn_worker(&jobs[t]) != NULL)
            failed = 1;
    if (attn_worker(&jobs[0]) != NULL)
        failed = 1;
    for (int32_t t = 1; t <= started; ++t) {
        void *ret = NULL;
        pthread_join(threads[t], &ret);
        if (ret != NULL)
            failed = 1;
    }
    free(jobs);
    free(threads);
    return failed ? -2 : n_threads;
}

/*
 * Attention for an arbitrary list of query rows over the paged pools.
 * Returns the number of threads used, or a negative value on bad arguments
 * or allocation failure.
 */
int32_t oracle_attention_rows(int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t head_dim, int32_t window, double softcap,
                              double scale, int32_t k_eq_v, int32_t block_size,
                              const uint16_t *q_rows, const int32_t *row_seq,
                              const int64_t *row_pos, int64_t n_rows,
                              const uint16_t *k_pool, const uint16_t *v_pool,
                              const int32_t *block_table,
                              int32_t max_blocks_per_seq, double *out,
                              double *lse, int32_t n_threads)
{
    return attention_rows(n_q_heads, n_kv_heads, head_dim, window, softcap, scale,
                          k_eq_v, block_size, q_rows, row_seq, row_pos, n_rows, k_pool,
                          v_pool, 0, NULL, NULL, NULL, NULL, block_table,
                          max_blocks_per_seq, out, lse, n_threads);
}

/* The same over FP8 pages: K_j = code * scale (V likewise; V reads the K
 * codes and scales when k_eq_v). */
int32_t oracle_attention_rows_fp8(int32_t n_q_heads, int32_t n_kv_heads,
                                  int32_t head_dim, int32_t window, double softcap,
                                  double scale, int32_t k_eq_v, int32_t block_size,
                                  const uint16_t *q_rows, const int32_t *row_seq,
                                  const int64_t *row_pos, int64_t n_rows,
                                  const uint8_t *k8, const uint8_t *v8,
                                  const float *k_scale, const float *v_scale,
                                  const int32_t *block_table,
                                  int32_t max_blocks_per_seq, double *out,
                                  double *lse, int32_t n_threads)
{
    return attention_rows(n_q_heads, n_kv_heads, head_dim, window, softcap, scale,
                          k_eq_v, block_size, q_rows, row_seq, row_pos, n_rows, NULL, NULL,
                          1, k8, v8, k_scale, v_scale, block_table, max_blocks_per_seq,
                          out, lse, n_threads);
}

/*
 * ---- pre-attention step: RMS-norm of q/k/v head vectors, proportional RoPE
 *
 * Per head vector x of length hd (all arithmetic in double):
 *   y_d = x_d / sqrt(mean_e(x_e^2) + eps) * w_d      (w_d = 1 when no weight)
 * (RMSNorm per head vector before RoPE: InfiniLM PR 581, Gemma-3 item 1; the
 * weights are the effective ones, the checkpoint's zero-centred w plus 1,
 * as that item's remapper loads them; v_norm: "MNN supports the full Gemma4
 * family", section 6.1.)
 * Then, for q and k only (V is not rotated: same page, section 6.2), the
 * proportional rotary embedding of "Gemma 4 model architecture analysis",
 * challenge 5: frequency i of the hd/2 pairs is theta^(-2i/hd) for
 * i < rope_angles and 0 beyond (the zero-padded, unrotated dims), so the
 * exponent's denominator is the head size, not the rotated size. Pair i
 * couples dims i and i + hd/2 (rotate-half form):
 *   out_i        = y_i cos(a_i) - y_{i+hd/2} sin(a_i)
 *   out_{i+hd/2} = y_{i+hd/2} cos(a_i) + y_i sin(a_i),   a_i = pos * freq_i
 */
void oracle_norm_rope_row(const uint16_t *x, int32_t hd, double eps,
                          const float *weight, int32_t rotate, double theta,
                          int32_t rope_angles, int64_t pos, double *out)
{
    double ss = 0.0;
    for (int32_t d = 0; d < hd; ++d) {
        double v = bf16_bits_to_double(x[d]);
        ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / (double)hd + eps);
    double *y = out; /* normalised in place, then rotated pair by pair */
    for (int32_t d = 0; d < hd; ++d)
        y[d] = bf16_bits_to_double(x[d]) * inv *
               (weight != NULL ? (double)weight[d] : 1.0);
    if (!rotate)
        return;
    int32_t half = hd / 2;
    for (int32_t i = 0; i < half; ++i) {
        double freq = (i < rope_angles)
                          ? pow(theta, -2.0 * (double)i / (double)hd)
                          : 0.0;
        double a = (double)pos * freq;
        double c = cos(a), s = sin(a);
        double lo = y[i], hi = y[i + half];
        y[i] = lo * c - hi * s;
        y[i + half] = hi * c + lo * s;
    }
}

/* Round a double to the nearest bf16 (ties to even); returns its bits. */
uint16_t oracle_to_bf16(double v)
{
    if (v != v)
        return 0x7FC0;
    int neg = signbit(v) != 0;
    double a = fabs(v);
    uint16_t sign = neg ? 0x8000 : 0;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e); /* a = f * 2^e, 0.5 <= f < 1 */
    /* quantum of a bf16 with this exponent (8 significant bits), never
       finer than the smallest subnormal 2^-133 */
    int qexp = e - 8;
    if (qexp < -133)
        qexp = -133;
    double n = nearbyint(ldexp(a, -qexp)); /* default rounding: ties to even */
    double r = ldexp(n, qexp);
    if (r > 3.3895313892515355e38) /* beyond the largest finite bf16 */
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/*
 * The whole pre-attention step of one layer for the new tokens of a batch:
 * token t of sequence b sits at position past_lens[b] + (t - cu_new[b]).
 * q_out[t][h] = rope(norm_q(q[t][h])); when k_rows is non-NULL (a layer that
 * owns its cache) k_rows[t][g] = rope(norm_k(k[t][g])) and, when v_rows is
 * non-NULL, v_rows[t][g] = norm_v(v[t][g]) (no rotation). Outputs in double;
 * writing them into pages is oracle_kv_cache_write's job, after rounding.
 */
void oracle_qkv_norm_rope(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *cu_new, const int32_t *past_lens,
                          int32_t n_seqs, int32_t n_q_heads, int32_t n_kv_heads,
                          int32_t hd, double eps, const float *q_w, const float *k_w,
                          const float *v_w, double theta, int32_t rope_angles,
                          double *q_out, double *k_rows, double *v_rows)
{
    for (int32_t b = 0; b < n_seqs; ++b) {
        for (int32_t t = cu_new[b]; t < cu_new[b + 1]; ++t) {
            int64_t pos = (int64_t)past_lens[b] + (t - cu_new[b]);
            for (int32_t h = 0; h < n_q_heads; ++h) {
                int64_t o = ((int64_t)t * n_q_heads + h) * hd;
                oracle_norm_rope_row(q + o, hd, eps, q_w, 1, theta, rope_angles, pos,
                                     q_out + o);
            }
            for (int32_t g = 0; g < n_kv_heads; ++g) {
                int64_t o = ((int64_t)t * n_kv_heads + g) * hd;
                if (k_rows != NULL)
                    oracle_norm_rope_row(k + o, hd, eps, k_w, 1, theta, rope_angles,
                                         pos, k_rows + o);
                if (v_rows != NULL)
                    oracle_norm_rope_row(v + o, hd, eps, v_w, 0, theta, rope_angles,
                                         pos, v_rows + o);
            }
        }
    }
}

/* oracle_to_bf16 over an array. */
void oracle_to_bf16_array(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_to_bf16(v[i]);
}

/* oracle_e4m3_encode / oracle_e4m3_decode over arrays. */
void oracle_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}
