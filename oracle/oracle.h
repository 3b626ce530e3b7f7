/*
 * oracle.h -- CPU fp64 oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg.  Shares nothing with the CUDA library.
 * Citations and readings are in oracle.c.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_RANGE = 3 };
enum { OR_F32 = 0, OR_BF16 = 1 };

/* Paged-attention problem description.  Pools are [num_blocks][block_size]
 * [num_kv_heads][head_dim]; q is [rows][num_heads][head_dim]; block_tables
 * is [num_seqs][max_blocks].  cu_seqlens_q may be NULL: one query row per
 * sequence (decode), row index = sequence index. */
typedef struct {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *cu_seqlens_q; /* nullable */
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int max_blocks;
    int num_blocks;
    int dtype;        /* OR_F32 or OR_BF16: q and both pools */
    double scale;
    int non_causal;   /* 1: every query row sees all context_lens[s] keys (encode) */
} or_problem;

long long or_num_blocks_needed(long long num_tokens, long long block_size);

int or_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                    const int32_t *seq_start, const int32_t *cu_seqlens_q,
                    int block_size, int num_blocks, int64_t *slot_mapping);

int or_reshape_and_cache(const void *key, const void *value,
                         int64_t key_stride_tok, int64_t value_stride_tok,
                         void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int dtype);

/* out: [rows][num_heads][head_dim] doubles */
int or_paged_attention(const or_problem *pr, double *out, int nthreads);

/* out: [nsel][head_dim] doubles for the (rows[k], heads[k]) pairs */
int or_paged_attention_rows(const or_problem *pr, const int32_t *rows,
                            const int32_t *heads, int nsel, double *out, int nthreads);

int or_attention_partial(const or_problem *pr, int s, int i, int h,
                         long long j_begin, long long j_end,
                         double *m, double *l, double *o);

int or_merge_partials(const double *m, const double *l, const double *o,
                      int nparts, int head_dim, double *out);

int or_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                   int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                   const int32_t *pairs, int num_pairs);

int or_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_ORACLE_H */
