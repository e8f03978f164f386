/*
 * pa_oracle.c - plain, slow, fp64 CPU oracle for attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link, load or
 * call this file: only the tests, the smoke check and the bench's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library; it takes
 * raw bf16 bit patterns (uint16) and int32 index arrays and returns fp64 results.
 *
 * What it computes, and where each step is defined:
 *
 *  store   "MinivLLM API docs - Attention", section store_kvcache: every token t
 *          whose slot_mapping[t] is not negative is copied to cache block
 *          slot // block_size, row slot % block_size; slot -1 marks a padding token
 *          that is skipped.  The vLLM learning book, "05 Attention Backends", Q&A 2,
 *          states the same indexing for the [2, num_blocks, block_size,
 *          num_kv_heads, head_size] cache (K half and V half).
 *  gather  "MinivLLM API docs - Attention", section paged_attention_decode
 *          (block_tables): logical block j of sequence i lives in physical block
 *          block_tables[i, j]; so key position p is row p % block_size of
 *          block block_tables[i, p // block_size].
 *  mask    "transformers continuous_batching/input_ouputs.py", build_attention_mask
 *          (docstring examples and the causal / sliding diagonals): the sq new
 *          queries are the last sq positions of the sk keys (bottom-right causal
 *          alignment), and a window of w keeps the w most recent keys including the
 *          query's own position.  The square case agrees with
 *          "vllm-npu 0.4.2, torch_sdpa.py", _make_sliding_window_bias (keys
 *          i-w+1..i).  Query row r of a sequence sits at absolute position
 *          sk - sq + r ("05 Attention Backends", section 4: seq_len = context_len +
 *          query_len).
 *  GQA     "vllm-npu 0.4.2, torch_sdpa.py", TorchSDPABackendImpl: num_queries_per_kv
 *          = num_heads / num_kv_heads and K/V are repeat_interleave'd, so query
 *          head h reads kv head h / num_queries_per_kv.
 *  softmax "MinivLLM API docs - Attention", sections flash_attention_prefill and
 *          paged_attention_decode: o = sum_j softmax_j(scale * q.k_j) v_j over the
 *          visible keys; scale is passed in final form (normally 1/sqrt(head_dim)).
 *
 *  state   "05 Attention Backends", section 7.1 (split-KV: each slice of a long
 *          context yields a partial result that is merged afterwards) and section 8
 *          (cascade attention: a shared prefix is attended once, each request's
 *          suffix separately, and the two are merged; mathematically equivalent).
 *          The partial result of a query over a subset J of its visible keys is the
 *          pair (o_J, lse_J): o_J = sum_{j in J} e^{s_j} v_j / sum_{j in J} e^{s_j}
 *          and lse_J = ln sum_{j in J} e^{s_j}, with s_j = scale * q.k_j.
 *  fp8     "vllm-npu 0.4.2 wheel diff", torch_sdpa.py / xformers.py: with an fp8 KV cache
 *          the cache write and the paged attention both take one kv_scale.  Reading
 *          taken: the cache holds FP8 E4M3 codes of x / kv_scale (the division in fp32,
 *          round to nearest even onto the E4M3 grid, finite values beyond 448 saturate
 *          to 448, NaN -> 0x7F) and attention reads code * kv_scale.
 *  merge   for disjoint subsets J_1..J_R of the visible keys, the attention over
 *          their union is o = sum_r e^{lse_r} o_r / sum_r e^{lse_r} and
 *          lse = ln sum_r e^{lse_r} (a subset with no keys has lse = -inf and
 *          contributes nothing).
 *
 * Everything is done in fp64 with no tiling, no online softmax and no reordering
 * beyond the plain definition: max, exp, sum, divide.
 *
 * Readings where the pages are silent (also listed in the design notes):
 *  - window <= 0 means "no window"; window == 1 keeps only the query's own key.
 *  - a query row with no visible key (only possible for seq_len == 0) yields zeros.
 *  - any negative slot is skipped (the pages use -1; other engines use -2).
 *
 * Return codes: 0 = ok, -1 = invalid argument, -2 = block index out of range,
 * -3 = out of memory.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ERANGE (-2)
#define ORACLE_ENOMEM (-3)

/* bf16 is the upper half of an IEEE binary32; widening to fp64 is exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double pa_oracle_bf16_to_double(uint16_t bits) { return bf16_bits_to_double(bits); }

/*
 * FP8 E4M3 (the "fn" variant: no infinities): sign, 4 exponent bits with bias 7, 3
 * mantissa bits.  Exponent field 0 holds the subnormals m/8 * 2^-6; S.1111.111 is NaN;
 * the largest finite magnitude is 1.75 * 2^8 = 448.
 */
double pa_oracle_fp8_e4m3_decode(uint8_t code)
{
    const int sign = code >> 7;
    const int e = (code >> 3) & 15;
    const int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = (m / 8.0) * ldexp(1.0, -6);
    else
        v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 value to x (ties to the even code, i.e. mantissa LSB 0), by search over
 * the 127 non-negative finite codes; finite |x| > 448 and +-inf saturate to +-448. */
uint8_t pa_oracle_fp8_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a > 448.0)
        return sign | 0x7E;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(pa_oracle_fp8_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/* store_kvcache into an FP8 E4M3 cache: code = encode(x / kv_scale), x the bf16 input
 * as fp32, the division in fp32. */
int pa_oracle_store_kvcache_fp8(const uint16_t *key, const uint16_t *value, uint8_t *k_cache,
                                uint8_t *v_cache, const int32_t *slot_mapping,
                                int64_t num_tokens, int64_t num_blocks, int block_size,
                                int num_kv_heads, int head_dim, float kv_scale)
{
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || !(kv_scale > 0.0f))
        return ORACLE_EINVAL;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size)
            return ORACLE_ERANGE;
        for (int64_t i = 0; i < row; ++i) {
            const float k = (float)bf16_bits_to_double(key[t * row + i]) / kv_scale;
            const float v = (float)bf16_bits_to_double(value[t * row + i]) / kv_scale;
            k_cache[slot * row + i] = pa_oracle_fp8_e4m3_encode(k);
            v_cache[slot * row + i] = pa_oracle_fp8_e4m3_encode(v);
        }
    }
    return ORACLE_OK;
}

/* One cache element as fp64: bf16 bits, or an FP8 E4M3 code times kv_scale. */
static double cache_elem(const void *cache, int fp8, double kv_scale, int64_t idx)
{
    if (fp8)
        return pa_oracle_fp8_e4m3_decode(((const uint8_t *)cache)[idx]) * kv_scale;
    return bf16_bits_to_double(((const uint16_t *)cache)[idx]);
}

/* ---------------------------------------------------------------- store --- */

int pa_oracle_store_kvcache(const uint16_t *key, const uint16_t *value,
                            uint16_t *k_cache, uint16_t *v_cache,
                            const int32_t *slot_mapping, int64_t num_tokens,
                            int64_t num_blocks, int block_size, int num_kv_heads,
                            int head_dim)
{
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return ORACLE_EINVAL;
    const int64_t row = (int64_t)num_kv_heads * head_dim; /* elements per token */
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue; /* padding token */
        const int64_t block_idx = slot / block_size;
        const int64_t block_offset = slot % block_size;
        if (block_idx >= num_blocks)
            return ORACLE_ERANGE;
        /* cache[block_idx][block_offset][:][:] = key[t][:][:] (and value). */
        const int64_t dst = (block_idx * block_size + block_offset) * row;
        for (int64_t e = 0; e < row; ++e) {
            k_cache[dst + e] = key[t * row + e];
            v_cache[dst + e] = value[t * row + e];
        }
    }
    return ORACLE_OK;
}

/* ----------------------------------------------------------------- mask --- */

/* Is key position j visible from a query at absolute position p? */
static int key_visible(int64_t p, int64_t j, int window)
{
    if (j > p)
        return 0; /* causal */
    if (window > 0 && j < p - window + 1)
        return 0; /* outside the window of `window` most recent keys */
    return 1;
}

/* allowed[r * sk + j] = 1 iff query row r (of sq new queries over sk keys) sees key j. */
int pa_oracle_mask(int sq, int sk, int window, uint8_t *allowed)
{
    if (sq < 0 || sk < 0 || sq > sk)
        return ORACLE_EINVAL;
    for (int r = 0; r < sq; ++r) {
        const int64_t p = (int64_t)sk - sq + r;
        for (int j = 0; j < sk; ++j)
            allowed[(int64_t)r * sk + j] = (uint8_t)key_visible(p, j, window);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------ attention --- */

/*
 * One query row, all heads, over the visible keys j >= key_begin.
 * q_row: [num_heads, head_dim] bf16 bits.  out: [num_heads, head_dim] fp64.
 * lse: [num_heads] fp64 (may be NULL): ln of the sum of e^{s_j} over those keys,
 * -inf when there are none (then the output row is zeros).
 * block_table_row: this sequence's row of the block table.  seq_len keys, query at
 * absolute position pos (pos < seq_len).  work: caller scratch of seq_len doubles
 * (NULL -> allocated here).
 */
static int attend_row_impl(double *out, double *lse, const uint16_t *q_row,
                           const void *k_cache, const void *v_cache, int fp8,
                           double kv_scale, const int32_t *block_table_row, int64_t seq_len,
                           int64_t pos, int64_t key_begin, int num_heads, int num_kv_heads,
                           int head_dim, int block_size, int64_t num_blocks, int window,
                           double scale, double *work)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        head_dim <= 0 || block_size <= 0 || seq_len < 0 || pos < 0 || key_begin < 0 ||
        (seq_len > 0 && pos >= seq_len))
        return ORACLE_EINVAL;
    const int group = num_heads / num_kv_heads; /* num_queries_per_kv */
    double *logits = work;
    int own = 0;
    if (logits == NULL && seq_len > 0) {
        logits = (double *)malloc((size_t)seq_len * sizeof(double));
        if (!logits)
            return ORACLE_ENOMEM;
        own = 1;
    }
    double *acc = (double *)malloc((size_t)head_dim * sizeof(double));
    if (!acc) {
        if (own)
            free(logits);
        return ORACLE_ENOMEM;
    }
    int rc = ORACLE_OK;
    for (int h = 0; h < num_heads && rc == ORACLE_OK; ++h) {
        const int kvh = h / group;
        const uint16_t *q = q_row + (int64_t)h * head_dim;
        /* logits s_j = scale * q . k_j for every visible key j */
        double m = -INFINITY;
        int64_t visible = 0;
        for (int64_t j = key_begin; j < seq_len; ++j) {
            if (!key_visible(pos, j, window))
                continue;
            const int64_t phys = block_table_row[j / block_size];
            if (phys < 0 || phys >= num_blocks) {
                rc = ORACLE_ERANGE;
                break;
            }
            const int64_t k0 =
                ((phys * block_size + j % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += bf16_bits_to_double(q[d]) * cache_elem(k_cache, fp8, kv_scale, k0 + d);
            logits[j] = scale * dot;
            if (logits[j] > m)
                m = logits[j];
            ++visible;
        }
        if (rc != ORACLE_OK)
            break;
        double *o = out + (int64_t)h * head_dim;
        if (visible == 0) {
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (lse)
                lse[h] = -INFINITY;
            continue;
        }
        /* softmax weights a_j = exp(s_j - m); o = sum_j a_j v_j / sum_j a_j */
        double denom = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc[d] = 0.0;
        for (int64_t j = key_begin; j < seq_len; ++j) {
            if (!key_visible(pos, j, window))
                continue;
            const int64_t phys = block_table_row[j / block_size];
            const int64_t v0 =
                ((phys * block_size + j % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;
            const double a = exp(logits[j] - m);
            denom += a;
            for (int d = 0; d < head_dim; ++d)
                acc[d] += a * cache_elem(v_cache, fp8, kv_scale, v0 + d);
        }
        for (int d = 0; d < head_dim; ++d)
            o[d] = acc[d] / denom;
        if (lse)
            lse[h] = m + log(denom);
    }
    free(acc);
    if (own)
        free(logits);
    return rc;
}

int pa_oracle_attend_row_state(double *out, double *lse, const uint16_t *q_row,
                               const uint16_t *k_cache, const uint16_t *v_cache,
                               const int32_t *block_table_row, int64_t seq_len, int64_t pos,
                               int64_t key_begin, int num_heads, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks, int window,
                               double scale, double *work)
{
    return attend_row_impl(out, lse, q_row, k_cache, v_cache, 0, 1.0, block_table_row,
                           seq_len, pos, key_begin, num_heads, num_kv_heads, head_dim,
                           block_size, num_blocks, window, scale, work);
}

/* One query row, all heads, over all its visible keys (attend_row_state from key 0). */
int pa_oracle_attend_row(double *out, const uint16_t *q_row, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table_row,
                         int64_t seq_len, int64_t pos, int num_heads, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, int window,
                         double scale, double *work)
{
    return pa_oracle_attend_row_state(out, NULL, q_row, k_cache, v_cache, block_table_row,
                                      seq_len, pos, 0, num_heads, num_kv_heads, head_dim,
                                      block_size, num_blocks, window, scale, work);
}

/*
 * Merge R partial results of the same rows (see "merge" above).  states:
 * [num_states, rows, head_dim], lses: [num_states, rows]; out: [rows, head_dim],
 * out_lse: [rows] (may be NULL).  Rows whose every part is empty get zeros / -inf.
 */
int pa_oracle_merge_states(double *out, double *out_lse, const double *states,
                           const double *lses, int num_states, int64_t rows, int head_dim)
{
    if (num_states <= 0 || rows < 0 || head_dim <= 0)
        return ORACLE_EINVAL;
    for (int64_t i = 0; i < rows; ++i) {
        double m = -INFINITY;
        for (int r = 0; r < num_states; ++r)
            if (lses[(int64_t)r * rows + i] > m)
                m = lses[(int64_t)r * rows + i];
        double *o = out + i * head_dim;
        for (int d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (m == -INFINITY) {
            if (out_lse)
                out_lse[i] = -INFINITY;
            continue;
        }
        double denom = 0.0;
        for (int r = 0; r < num_states; ++r) {
            const double w = exp(lses[(int64_t)r * rows + i] - m);
            denom += w;
            const double *src = states + ((int64_t)r * rows + i) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * src[d];
        }
        for (int d = 0; d < head_dim; ++d)
            o[d] /= denom;
        if (out_lse)
            out_lse[i] = m + log(denom);
    }
    return ORACLE_OK;
}

/* Work list shared by the threads of pa_oracle_paged_attention. */
typedef struct {
    double *out;
    const uint16_t *q;
    const void *k_cache, *v_cache;
    int fp8;
    double kv_scale;
    const int32_t *cu_seqlens_q, *seq_lens, *block_table;
    int64_t max_num_blocks;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size, window;
    int64_t num_blocks;
    double scale;
    int64_t total_rows;
    int64_t max_seq_len;
    int64_t next_row; /* guarded by lock */
    pthread_mutex_t lock;
    int rc; /* first error, guarded by lock */
} oracle_job;

/* Sequence owning packed query row t: cu_seqlens_q is non-decreasing. */
static int seq_of_row(const int32_t *cu, int num_seqs, int64_t t)
{
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    double *work = NULL;
    if (job->max_seq_len > 0) {
        work = (double *)malloc((size_t)job->max_seq_len * sizeof(double));
        if (!work) {
            pthread_mutex_lock(&job->lock);
            if (job->rc == ORACLE_OK)
                job->rc = ORACLE_ENOMEM;
            pthread_mutex_unlock(&job->lock);
            return NULL;
        }
    }
    const int64_t row_elems = (int64_t)job->num_heads * job->head_dim;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        const int64_t t = job->next_row++;
        const int failed = job->rc != ORACLE_OK;
        pthread_mutex_unlock(&job->lock);
        if (t >= job->total_rows || failed)
            break;
        const int i = seq_of_row(job->cu_seqlens_q, job->num_seqs, t);
        const int64_t sq = job->cu_seqlens_q[i + 1] - job->cu_seqlens_q[i];
        const int64_t sk = job->seq_lens[i];
        const int64_t r = t - job->cu_seqlens_q[i];
        const int64_t pos = sk - sq + r; /* bottom-right alignment */
        const int rc = attend_row_impl(
            job->out + t * row_elems, NULL, job->q + t * row_elems, job->k_cache,
            job->v_cache, job->fp8, job->kv_scale,
            job->block_table + (int64_t)i * job->max_num_blocks, sk, pos, 0, job->num_heads,
            job->num_kv_heads, job->head_dim, job->block_size, job->num_blocks,
            job->window, job->scale, work);
        if (rc != ORACLE_OK) {
            pthread_mutex_lock(&job->lock);
            if (job->rc == ORACLE_OK)
                job->rc = rc;
            pthread_mutex_unlock(&job->lock);
        }
    }
    free(work);
    return NULL;
}

/*
 * Paged attention for a packed batch.  Sequence i owns query rows
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) and seq_lens[i] keys; decode is the case
 * cu_seqlens_q = 0, 1, ..., num_seqs.  q, out: [total_rows, num_heads, head_dim].
 * block_table: [num_seqs, max_num_blocks].  num_threads <= 0 -> all online CPUs.
 */
static int paged_attention_impl(double *out, const uint16_t *q, const void *k_cache,
                                const void *v_cache, int fp8, double kv_scale,
                                const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                                const int32_t *block_table, int64_t max_num_blocks,
                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int64_t num_blocks, int window, double scale,
                                int num_threads)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (num_seqs == 0)
        return ORACLE_OK;
    int64_t max_seq_len = 0;
    for (int i = 0; i < num_seqs; ++i) {
        const int64_t sq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        const int64_t sk = seq_lens[i];
        if (sq < 0 || sk < 0 || sq > sk)
            return ORACLE_EINVAL;
        if ((sk + block_size - 1) / block_size > max_num_blocks)
            return ORACLE_EINVAL;
        if (sk > max_seq_len)
            max_seq_len = sk;
    }
    oracle_job job;
    job.out = out;
    job.q = q;
    job.k_cache = k_cache;
    job.v_cache = v_cache;
    job.fp8 = fp8;
    job.kv_scale = kv_scale;
    job.cu_seqlens_q = cu_seqlens_q;
    job.seq_lens = seq_lens;
    job.block_table = block_table;
    job.max_num_blocks = max_num_blocks;
    job.num_seqs = num_seqs;
    job.num_heads = num_heads;
    job.num_kv_heads = num_kv_heads;
    job.head_dim = head_dim;
    job.block_size = block_size;
    job.window = window;
    job.num_blocks = num_blocks;
    job.scale = scale;
    job.total_rows = cu_seqlens_q[num_seqs]; /* rows run from cu[0] to cu[num_seqs] */
    job.max_seq_len = max_seq_len;
    job.next_row = cu_seqlens_q[0];
    job.rc = ORACLE_OK;
    pthread_mutex_init(&job.lock, NULL);

    if (num_threads <= 0) {
        const long n = sysconf(_SC_NPROCESSORS_ONLN);
        num_threads = n > 0 ? (int)n : 1;
    }
    if (num_threads > 1024)
        num_threads = 1024;
    pthread_t *threads = (pthread_t *)malloc((size_t)num_threads * sizeof(pthread_t));
    if (!threads) {
        pthread_mutex_destroy(&job.lock);
        return ORACLE_ENOMEM;
    }
    int started = 0;
    for (int n = 1; n < num_threads; ++n) {
        if (pthread_create(&threads[n], NULL, oracle_worker, &job) != 0)
            break;
        ++started;
    }
    oracle_worker(&job); /* the calling thread works too */
    for (int n = 1; n <= started; ++n)
        pthread_join(threads[n], NULL);
    free(threads);
    pthread_mutex_destroy(&job.lock);
    return job.rc;
}

int pa_oracle_paged_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *cu_seqlens_q,
                              const int32_t *seq_lens, const int32_t *block_table,
                              int64_t max_num_blocks, int num_seqs, int num_heads,
                              int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, int window, double scale,
                              int num_threads)
{
    return paged_attention_impl(out, q, k_cache, v_cache, 0, 1.0, cu_seqlens_q, seq_lens,
                                block_table, max_num_blocks, num_seqs, num_heads,
                                num_kv_heads, head_dim, block_size, num_blocks, window, scale,
                                num_threads);
}

/* The same over an FP8 E4M3 cache read as code * kv_scale. */
int pa_oracle_paged_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                                  const uint8_t *v_cache, const int32_t *cu_seqlens_q,
                                  const int32_t *seq_lens, const int32_t *block_table,
                                  int64_t max_num_blocks, int num_seqs, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, int window, double scale,
                                  double kv_scale, int num_threads)
{
    if (!(kv_scale > 0.0))
        return ORACLE_EINVAL;
    return paged_attention_impl(out, q, k_cache, v_cache, 1, kv_scale, cu_seqlens_q, seq_lens,
                                block_table, max_num_blocks, num_seqs, num_heads,
                                num_kv_heads, head_dim, block_size, num_blocks, window, scale,
                                num_threads);
}

/* Number of threads pa_oracle_paged_attention uses for num_threads <= 0. */
int pa_oracle_default_threads(void)
{
    const long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
