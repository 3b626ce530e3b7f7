/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the paged KV-cache
 * hot path (block count, slot mapping, cache write, paged attention, split
 * merge).
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Arithmetic: every floating-point quantity is carried in IEEE double.  bf16
 * and fp32 inputs widen to double exactly, so the only rounding is fp64's.
 * There is no blocking, no online softmax and no split inside an attention
 * row: each row is the textbook definition, with keys taken in logical order.
 *
 * Sources (page title, section):
 *  [iitog]  "vLLM изнутри: как устроен движок для быстрого инференса LLM"
 *           -- allocate_slots paragraph (16 tokens per block, a 17-token
 *           prefill needs ceil(17/16) = 2 blocks); model-runner paragraph
 *           (slot map built during input preparation; all sequences of the
 *           batch are concatenated into one super-sequence and masks plus
 *           positions keep each sequence on its own tokens); decode reads
 *           the KV of earlier tokens from the cache.
 *  [kwkr]   "vLLM：颠覆大模型推理的高效API服务引擎深度解析" -- §1.2 (block =
 *           fixed number of tokens, block table maps logical block i to a
 *           physical block and records its fill count), §1.3 (one shared
 *           pre-allocated pool; a new token's K/V vectors are stored into
 *           its physical block; attention gathers the scattered blocks into
 *           a logically contiguous KV through the block table; physical
 *           blocks may be referenced read-only by several block tables).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *  - slot of the token at logical position p of sequence s is
 *      block_tables[s][p / B] * B + p % B
 *    over a pool laid out [num_blocks][B][num_kv_heads][head_dim];
 *  - a negative slot means "no write" (padding sentinel);
 *  - context_lens counts every token the query may see, including the ones
 *    being written in this step; query i of a sequence with q_len new tokens
 *    sits at position ctx - q_len + i and sees keys 0..that position;
 *  - q-head h uses kv-head h / (num_heads / num_kv_heads);
 *  - encode-only attention (the embedding workload of "vLLMつかったら、
 *    ベクトル検索サーバーが高速化して安定性も向上した": vector search only
 *    encodes) drops the causal mask: every query row of a sequence sees all
 *    of that sequence's context_lens[s] keys, and still no other sequence's.
 *
 * Parity pins: every function is pinned by tests (worked examples printed
 * on the pages, closed forms, invariants, fp64 torch SDPA, brute force); see
 * tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

/* ---- element access: widen one stored element to double (exact) -------- */
static double load_elem(const void *base, int64_t idx, int dtype)
{
    if (dtype == OR_F32) {
        return (double)((const float *)base)[idx];
    }
    /* bf16: the stored 16 bits are the top half of an IEEE binary32. */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static int elem_bytes(int dtype)
{
    return dtype == OR_F32 ? 4 : (dtype == OR_BF16 ? 2 : 0);
}

/* ---- a1: number of blocks a run of tokens needs ([iitog]) --------------- */
long long or_num_blocks_needed(long long num_tokens, long long block_size)
{
    if (block_size <= 0 || num_tokens < 0) return -1;
    long long n = num_tokens / block_size;
    if (n * block_size < num_tokens) n += 1; /* round up */
    return n;
}

/* ---- a2: slot mapping ([iitog] model runner, [kwkr] §1.2-1.3) ----------- */
int or_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                    const int32_t *seq_start, const int32_t *cu_seqlens_q,
                    int block_size, int num_blocks, int64_t *slot_mapping)
{
    if (num_seqs < 0 || max_blocks <= 0 || block_size <= 0) return OR_ERR_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        int first = cu_seqlens_q[s];
        int last = cu_seqlens_q[s + 1];
        if (last < first || seq_start[s] < 0) return OR_ERR_ARG;
        for (int t = first; t < last; ++t) {
            long long pos = (long long)seq_start[s] + (t - first);
            long long logical_block = pos / block_size;
            long long offset = pos % block_size;
            if (logical_block >= max_blocks) return OR_ERR_RANGE;
            int32_t phys = block_tables[(int64_t)s * max_blocks + logical_block];
            if (phys < 0 || phys >= num_blocks) return OR_ERR_RANGE;
            slot_mapping[t] = (int64_t)phys * block_size + offset;
        }
    }
    return OR_OK;
}

/* ---- a3: cache write ([kwkr] §1.3 "store the new token's KV") ----------- */
int or_reshape_and_cache(const void *key, const void *value,
                         int64_t key_stride_tok, int64_t value_stride_tok,
                         void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int dtype)
{
    int eb = elem_bytes(dtype);
    if (eb == 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return OR_ERR_ARG;
    int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    int64_t pool_slots = (int64_t)num_blocks * block_size;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;            /* padding: nothing to store */
        if (slot >= pool_slots) return OR_ERR_RANGE;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        /* pool row (block, offset) holds all kv-heads of one token */
        int64_t dst_elem = (block * block_size + offset) * row_elems;
        memcpy((char *)k_cache + dst_elem * eb,
               (const char *)key + (int64_t)t * key_stride_tok * eb, row_elems * eb);
        memcpy((char *)v_cache + dst_elem * eb,
               (const char *)value + (int64_t)t * value_stride_tok * eb, row_elems * eb);
    }
    return OR_OK;
}

/* ---- a4/a6: paged attention -------------------------------------------- */

/* Where the logical key j of sequence s, kv-head g, starts in the pool,
 * reached through the block table ([kwkr] §1.3 gather). */
static int key_row_offset(const or_problem *pr, int s, int64_t j, int g,
                          int64_t *elem_off)
{
    int64_t logical_block = j / pr->block_size;
    int64_t offset = j % pr->block_size;
    if (logical_block >= pr->max_blocks) return OR_ERR_RANGE;
    int32_t phys = pr->block_tables[(int64_t)s * pr->max_blocks + logical_block];
    if (phys < 0 || phys >= pr->num_blocks) return OR_ERR_RANGE;
    *elem_off = (((int64_t)phys * pr->block_size + offset) * pr->num_kv_heads + g)
                * pr->head_dim;
    return OR_OK;
}

/* Query rows of sequence s: [first, first + q_len).  Without cu_seqlens_q
 * every sequence has exactly one query row (decode), row index = s. */
static void query_rows(const or_problem *pr, int s, int *first, int *q_len)
{
    if (pr->cu_seqlens_q) {
        *first = pr->cu_seqlens_q[s];
        *q_len = pr->cu_seqlens_q[s + 1] - pr->cu_seqlens_q[s];
    } else {
        *first = s;
        *q_len = 1;
    }
}

static int check_sequence(const or_problem *pr, int s, int *ctx, int *q_len, int *first)
{
    query_rows(pr, s, first, q_len);
    *ctx = pr->context_lens[s];
    if (*ctx <= 0) return OR_ERR_RANGE;
    if ((int64_t)*ctx > (int64_t)pr->max_blocks * pr->block_size) return OR_ERR_RANGE;
    if (*q_len < 0 || *q_len > *ctx) return OR_ERR_RANGE;
    return OR_OK;
}

/* Logits x_j = scale * <q, k_j> for keys j in [j_begin, j_end) of query row
 * `row` (sequence s), q-head h.  Fills x[0 .. j_end-j_begin). */
static int logits(const or_problem *pr, int s, int row, int h,
                  int64_t j_begin, int64_t j_end, double *x)
{
    int group = pr->num_heads / pr->num_kv_heads;
    int g = h / group; /* kv-head serving q-head h */
    int64_t q_off = ((int64_t)row * pr->num_heads + h) * pr->head_dim;
    for (int64_t j = j_begin; j < j_end; ++j) {
        int64_t k_off;
        int rc = key_row_offset(pr, s, j, g, &k_off);
        if (rc) return rc;
        double dot = 0.0;
        for (int d = 0; d < pr->head_dim; ++d)
            dot += load_elem(pr->q, q_off + d, pr->dtype) *
                   load_elem(pr->k_cache, k_off + d, pr->dtype);
        x[j - j_begin] = pr->scale * dot;
    }
    return OR_OK;
}

/* One (query row, q-head): o = sum_j softmax(x)_j v_j over keys 0..pos. */
static int attend_one(const or_problem *pr, int s, int i, int h, double *o)
{
    int ctx, q_len, first;
    int rc = check_sequence(pr, s, &ctx, &q_len, &first);
    if (rc) return rc;
    if (i < 0 || i >= q_len) return OR_ERR_ARG;
    int64_t pos = (int64_t)ctx - q_len + i;   /* position of this query */
    int64_t n = pos + 1;                      /* keys 0..pos are visible */
    if (pr->non_causal) n = ctx;              /* encode: the whole sequence */
    double *x = (double *)malloc((size_t)n * sizeof(double));
    if (!x) return OR_ERR_ARG;
    rc = logits(pr, s, first + i, h, 0, n, x);
    if (rc) { free(x); return rc; }

    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) if (x[j] > mx) mx = x[j];
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) { x[j] = exp(x[j] - mx); z += x[j]; }

    int g = h / (pr->num_heads / pr->num_kv_heads);
    for (int d = 0; d < pr->head_dim; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t v_off;
        rc = key_row_offset(pr, s, j, g, &v_off);
        if (rc) { free(x); return rc; }
        double w = x[j] / z;
        for (int d = 0; d < pr->head_dim; ++d)
            o[d] += w * load_elem(pr->v_cache, v_off + d, pr->dtype);
    }
    free(x);
    return OR_OK;
}

static int check_problem(const or_problem *pr)
{
    if (!pr || !pr->q || !pr->k_cache || !pr->v_cache || !pr->block_tables ||
        !pr->context_lens) return OR_ERR_ARG;
    if (elem_bytes(pr->dtype) == 0) return OR_ERR_ARG;
    if (pr->num_heads <= 0 || pr->num_kv_heads <= 0 ||
        pr->num_heads % pr->num_kv_heads != 0) return OR_ERR_ARG;
    if (pr->head_dim <= 0 || pr->block_size <= 0 || pr->max_blocks <= 0 ||
        pr->num_blocks <= 0 || pr->num_seqs < 0) return OR_ERR_ARG;
    return OR_OK;
}

int or_paged_attention(const or_problem *pr, double *out, int nthreads)
{
    int rc = check_problem(pr);
    if (rc) return rc;
    /* enumerate (sequence, query index) pairs in row order */
    int total_rows = 0;
    for (int s = 0; s < pr->num_seqs; ++s) {
        int ctx, q_len, first;
        rc = check_sequence(pr, s, &ctx, &q_len, &first);
        if (rc) return rc;
        total_rows += q_len;
    }
    int *row_seq = (int *)malloc(sizeof(int) * (size_t)(total_rows > 0 ? total_rows : 1));
    int *row_idx = (int *)malloc(sizeof(int) * (size_t)(total_rows > 0 ? total_rows : 1));
    int *row_out = (int *)malloc(sizeof(int) * (size_t)(total_rows > 0 ? total_rows : 1));
    if (!row_seq || !row_idx || !row_out) { free(row_seq); free(row_idx); free(row_out); return OR_ERR_ARG; }
    int k = 0;
    for (int s = 0; s < pr->num_seqs; ++s) {
        int ctx, q_len, first;
        check_sequence(pr, s, &ctx, &q_len, &first);
        for (int i = 0; i < q_len; ++i) { row_seq[k] = s; row_idx[k] = i; row_out[k] = first + i; ++k; }
    }
    int64_t pairs = (int64_t)total_rows * pr->num_heads;
    int err = OR_OK;
    (void)nthreads;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : 1;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nt)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        int r = (int)(p / pr->num_heads);
        int h = (int)(p % pr->num_heads);
        double *o = out + ((int64_t)row_out[r] * pr->num_heads + h) * pr->head_dim;
        int e = attend_one(pr, row_seq[r], row_idx[r], h, o);
        if (e) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = e;
        }
    }
    free(row_seq); free(row_idx); free(row_out);
    return err;
}

/* Selected (query row, q-head) pairs only; out is [nsel][head_dim].  Used to
 * check full-size workloads on a sample of outputs. */
int or_paged_attention_rows(const or_problem *pr, const int32_t *rows,
                            const int32_t *heads, int nsel, double *out, int nthreads)
{
    int rc = check_problem(pr);
    if (rc) return rc;
    int err = OR_OK;
    (void)nthreads;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int k = 0; k < nsel; ++k) {
        /* find the sequence that owns query row rows[k] */
        int s_found = -1, i_found = -1;
        for (int s = 0; s < pr->num_seqs; ++s) {
            int first, q_len;
            query_rows(pr, s, &first, &q_len);
            if (rows[k] >= first && rows[k] < first + q_len) { s_found = s; i_found = rows[k] - first; break; }
        }
        int e = OR_ERR_ARG;
        if (s_found >= 0 && heads[k] >= 0 && heads[k] < pr->num_heads)
            e = attend_one(pr, s_found, i_found, heads[k], out + (int64_t)k * pr->head_dim);
        if (e) {
#ifdef _OPENMP
#pragma omp critical
#endif
            err = e;
        }
    }
    return err;
}

/* ---- a5: split partials and their merge -------------------------------- */

/* Partial state of one query row over the key range [j_begin, j_end):
 *   m = max x_j,  l = sum exp(x_j - m),  o[d] = sum exp(x_j - m) v_j[d]. */
int or_attention_partial(const or_problem *pr, int s, int i, int h,
                         long long j_begin, long long j_end,
                         double *m, double *l, double *o)
{
    int rc = check_problem(pr);
    if (rc) return rc;
    int ctx, q_len, first;
    rc = check_sequence(pr, s, &ctx, &q_len, &first);
    if (rc) return rc;
    int64_t pos = (int64_t)ctx - q_len + i;
    if (i < 0 || i >= q_len || j_begin < 0 || j_end > pos + 1 || j_end <= j_begin)
        return OR_ERR_ARG;
    int64_t n = j_end - j_begin;
    double *x = (double *)malloc((size_t)n * sizeof(double));
    if (!x) return OR_ERR_ARG;
    rc = logits(pr, s, first + i, h, j_begin, j_end, x);
    if (rc) { free(x); return rc; }
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) if (x[j] > mx) mx = x[j];
    double z = 0.0;
    int g = h / (pr->num_heads / pr->num_kv_heads);
    for (int d = 0; d < pr->head_dim; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double w = exp(x[j] - mx);
        z += w;
        int64_t v_off;
        rc = key_row_offset(pr, s, j_begin + j, g, &v_off);
        if (rc) { free(x); return rc; }
        for (int d = 0; d < pr->head_dim; ++d)
            o[d] += w * load_elem(pr->v_cache, v_off + d, pr->dtype);
    }
    *m = mx;
    *l = z;
    free(x);
    return OR_OK;
}

/* Merge: M = max m_i, L = sum l_i e^{m_i - M}, out = sum e^{m_i - M} o_i / L. */
int or_merge_partials(const double *m, const double *l, const double *o,
                      int nparts, int head_dim, double *out)
{
    if (nparts <= 0 || head_dim <= 0) return OR_ERR_ARG;
    double big = -INFINITY;
    for (int i = 0; i < nparts; ++i) if (m[i] > big) big = m[i];
    double total = 0.0;
    for (int i = 0; i < nparts; ++i) total += l[i] * exp(m[i] - big);
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int i = 0; i < nparts; ++i)
            acc += exp(m[i] - big) * o[(int64_t)i * head_dim + d];
        out[d] = acc / total;
    }
    return OR_OK;
}

/* ---- block copy: swap in/out, fork, pack/unpack ([kwkr] §1.3 swap space,
 * §2.2 the block manager moves inactive physical blocks to host memory and
 * back; §1.3 blocks shared by several requests).  For each pair (src, dst),
 * the whole block src of the source pools is copied byte for byte to block
 * dst of the destination pools.  A negative src or dst skips the pair. */
int or_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                   int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                   const int32_t *pairs, int num_pairs)
{
    if (block_bytes <= 0 || num_pairs < 0) return OR_ERR_ARG;
    for (int i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || dst < 0) continue;
        if (src >= src_num_blocks || dst >= dst_num_blocks) return OR_ERR_RANGE;
        memcpy((char *)dst_k + (int64_t)dst * block_bytes,
               (const char *)src_k + (int64_t)src * block_bytes, (size_t)block_bytes);
        memcpy((char *)dst_v + (int64_t)dst * block_bytes,
               (const char *)src_v + (int64_t)src * block_bytes, (size_t)block_bytes);
    }
    return OR_OK;
}

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
