/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged KV-cache library: slot mapping,
 * KV-cache write ("reshape_and_cache"), paged decode attention with a split-KV
 * reduction, and varlen paged prefill over a mixed prefill + decode batch.
 *
 * Sources for what each call computes (page title, section):
 *  [iitog] "vLLM изнутри: как устроен движок для быстрого инференса LLM":
 *          allocate_slots paragraph (blocks of 16 tokens, ceil(17/16) = 2);
 *          model-runner paragraph (slot map built while preparing inputs; the
 *          batch is one concatenated super-sequence in which masks and
 *          positions keep every sequence on its own tokens; prefill is
 *          compute-bound, decode reads earlier tokens' KV from the cache and
 *          is memory-bound).
 *  [kwkr]  "vLLM：颠覆大模型推理的高效API服务引擎深度解析": §1.2 (fixed-size
 *          blocks, per-request block table from logical to physical blocks),
 *          §1.3 (one pre-allocated pool shared by all requests; a new token's
 *          K/V vectors are stored into its physical block; attention gathers
 *          the scattered blocks into a logically contiguous KV through the
 *          block table; blocks may be referenced read-only by several block
 *          tables, e.g. a shared system prompt).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, except the
 *    host output of pa_get_device_status.  The library never allocates or
 *    frees device memory; scratch comes from the caller's `workspace`, sized
 *    by the matching *_workspace_size call.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Only pa_get_device_status synchronises.
 *  - Argument errors are found on the host before any launch and returned
 *    as a pa_status; nothing is launched then.
 *  - Data-dependent range errors (a block id outside [0, num_blocks), a slot
 *    outside the pool, a context length <= 0 or beyond max_blocks*block_size)
 *    are recorded into *dev_status (when dev_status != NULL) as
 *    PA_ERR_OUT_OF_RANGE by the first failing thread; the offending element
 *    is skipped, no out-of-bounds access is made and nothing traps.  Rows of
 *    `out` whose sequence had such an error are unspecified (a context length
 *    error leaves the row untouched).  A bounded wait inside a kernel that
 *    runs out records PA_ERR_TIMEOUT the same way.
 *  - Layouts (all row-major, contiguous unless a stride is given):
 *      pools        k_cache, v_cache: [num_blocks][block_size][num_kv_heads][head_dim]
 *      block_tables int32 [num_seqs][max_blocks]; entries past a sequence's
 *                   last block are never read
 *      q, out       [rows][num_heads][head_dim]
 *      key, value   [num_tokens][num_kv_heads][head_dim], token stride given
 *      slot_mapping int64 [num_tokens]
 *  - q-head h reads kv-head h / (num_heads / num_kv_heads) (MHA, GQA, MQA).
 *  - Supported: block_size 8, 16 or 32 for the attention calls (any block
 *    size >= 1 for pa_compute_slot_mapping and pa_reshape_and_cache); head_dim
 *    64 or 128; pa_dtype F32 or BF16 for q, key/value, pools and out alike
 *    (fp32 accumulation in every case).  Anything else returns
 *    PA_ERR_UNSUPPORTED.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
    PA_ERR_UNSUPPORTED = 2,  /* a valid shape this build does not implement */
    PA_ERR_OUT_OF_RANGE = 3, /* data-dependent index error (device status) */
    PA_ERR_WORKSPACE = 4,    /* workspace missing or too small */
    PA_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    PA_ERR_TIMEOUT = 6       /* a bounded in-kernel wait ran out (device status) */
} pa_status;

typedef enum { PA_DTYPE_F32 = 0, PA_DTYPE_BF16 = 1 } pa_dtype;

/* Human-readable name of a status code.  Never NULL. */
PA_API const char *pa_status_string(int status);

/* Library ABI version (major * 100 + minor). */
PA_API int pa_version(void);

/*
 * Number of blocks that hold num_tokens tokens: ceil(num_tokens / block_size)
 * ([iitog] allocate_slots: 17 new tokens at block size 16 need 2 blocks).
 * Host-only.  Returns -1 when num_tokens < 0 or block_size <= 0.
 */
PA_API int pa_num_blocks_needed(int num_tokens, int block_size);

/*
 * Slot mapping ([iitog] model runner builds the slot map; [kwkr] §1.2-1.3):
 * for new token j of sequence s (cu_seqlens_q[s] <= j < cu_seqlens_q[s+1]),
 * at logical position p = seq_start[s] + (j - cu_seqlens_q[s]),
 *     slot_mapping[j] = block_tables[s][p / block_size] * block_size
 *                       + p % block_size.
 *  block_tables  device int32 [num_seqs][max_blocks]
 *  seq_start     device int32 [num_seqs]: tokens already cached before the step
 *  cu_seqlens_q  device int32 [num_seqs + 1], cu_seqlens_q[0] = 0,
 *                cu_seqlens_q[num_seqs] = total_new
 *  slot_mapping  device int64 [total_new] (output)
 * A token whose logical block is >= max_blocks or whose table entry lies
 * outside [0, num_blocks) gets slot -1 and sets PA_ERR_OUT_OF_RANGE.
 */
PA_API pa_status pa_compute_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                                  const int32_t *seq_start, const int32_t *cu_seqlens_q,
                                  int total_new, int block_size, int num_blocks,
                                  int64_t *slot_mapping, int32_t *dev_status,
                                  pa_stream_t stream);

/*
 * KV-cache write ([kwkr] §1.3: store the new token's K/V vectors into its
 * physical block):  for t < num_tokens with slot = slot_mapping[t] >= 0,
 *     k_cache[slot / B][slot % B][:][:] = key[t][:][:]   (and v_cache / value).
 * Rows are copied bit for bit.  A negative slot is skipped (padding).  A slot
 * >= num_blocks * block_size is skipped and sets PA_ERR_OUT_OF_RANGE.
 *  key, value      device [num_tokens][num_kv_heads][head_dim]; the token
 *                  stride (in elements) may exceed num_kv_heads*head_dim so a
 *                  fused QKV projection output can be passed directly
 *  k_cache/v_cache device pools (see layouts above), written in place
 * Precondition (not checked on the device): live slots are pairwise distinct
 * and do not lie in a block that another sequence shares read-only.
 */
PA_API pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t key_stride_tok,
                               int64_t value_stride_tok, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                               int32_t *dev_status, pa_stream_t stream);

/*
 * Workspace bytes pa_decode needs for these sizes (0 is never returned).
 * Independent of the data; depends only on the arguments.
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks);

/*
 * Paged decode attention ([kwkr] §1.3 attention through the block table;
 * [iitog] decode reads earlier tokens' KV from the cache): one query row per
 * sequence, at position context_lens[s] - 1, for each q-head h with kv-head
 * g = h / (num_heads / num_kv_heads):
 *     x_j = scale * <q[s][h], K_s[j][g]>,  j < context_lens[s],
 *     out[s][h] = sum_j softmax(x)_j V_s[j][g],
 * where K_s[j] = k_cache[block_tables[s][j / B]][j % B] (same for V).
 * context_lens counts the new token, which pa_reshape_and_cache has already
 * written.  Long contexts are split across thread blocks; inside the same
 * kernel, the warp that stores a sequence's last piece merges the pieces
 * with the log-sum-exp rule
 *     M = max m_i,  L = sum l_i e^{m_i - M},  o = sum e^{m_i - M} o_i / L.
 *  out          device [num_seqs][num_heads][head_dim], dtype of q
 *  q            device [num_seqs][num_heads][head_dim]
 *  scale        the fp32 softmax scale, normally 1/sqrtf(head_dim)
 *  workspace    device scratch of >= pa_decode_workspace_size(...) bytes,
 *               16-byte aligned; its contents on entry do not matter
 * Results are deterministic: they depend on context_lens and the device's SM
 * count, never on which physical blocks hold the data.
 */
PA_API pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                    int num_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_blocks, int num_blocks, float scale, pa_dtype dtype,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status,
                    pa_stream_t stream);

/*
 * Decode without a caller workspace.  The paper has no counterpart: this is a
 * convenience for callers that cannot allocate device memory -- for example a
 * plugin interface that only hands over input and output pointers, or a
 * serving process whose memory pool has already claimed the device's free
 * memory for the KV cache.  Same arguments and results as pa_decode, minus
 * the workspace.
 *
 * The scratch is a fixed PA_STATIC_SCRATCH_BYTES (24 MiB) array inside the
 * library: every GPU that loads the library holds it until the process
 * exits.  Arguments are checked exactly as pa_decode checks them, with the
 * same status codes.  Then, for a call that takes the split decode (bf16,
 * head_dim 64/128, the shapes pa_decode serves with scratch), a problem whose
 * pa_decode_workspace_size(...) exceeds the array returns PA_ERR_WORKSPACE
 * before anything is launched; calls that take the CUDA-core kernel use no
 * scratch and have no such limit.  The call allocates nothing.
 * The first call on each device, and the first after a cudaDeviceReset
 * (which makes a new CUDA context), looks up the array's device address with
 * a synchronous CUDA runtime call, so make that call before any stream
 * capture.  Every call shares the one array and leaves its last contents
 * there; nothing in it has to start at zero.  Calls that can overlap on the
 * GPU (different streams, or several devices' threads targeting one device)
 * race on the array: serialise them.
 */
#define PA_STATIC_SCRATCH_BYTES ((size_t)24 << 20)
PA_API pa_status pa_decode_static_scratch(void *out, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int num_seqs,
                                          int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int max_blocks, int num_blocks,
                                          float scale, pa_dtype dtype, int32_t *dev_status,
                                          pa_stream_t stream);

/*
 * One decode step in one call: exactly pa_compute_slot_mapping, then
 * pa_reshape_and_cache of the step's new tokens, then pa_decode (same
 * arguments, same results; slot_mapping is written as an output).  On the
 * fast path (bf16, head_dim 64/128, 16-byte aligned rows and strides) the slot
 * mapping and the cache write run inside the decode plan kernel, saving two
 * launches and their dependent memory round trips; otherwise the three calls
 * run one after the other.
 *  key, value     device [total_new][num_kv_heads][head_dim], token strides given
 *  seq_start      device int32 [num_seqs]: tokens cached before this step
 *  cu_seqlens_new device int32 [num_seqs + 1]: offsets of the new tokens
 *  workspace      >= pa_decode_workspace_size(...) bytes
 * Each query row s attends to context_lens[s] tokens, which must include the
 * tokens this call writes.
 */
PA_API pa_status pa_decode_step(void *out, const void *q, const void *key, const void *value,
                                int64_t key_stride_tok, int64_t value_stride_tok, void *k_cache,
                                void *v_cache, const int32_t *block_tables,
                                const int32_t *context_lens, const int32_t *seq_start,
                                const int32_t *cu_seqlens_new, int total_new,
                                int64_t *slot_mapping, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size, int max_blocks,
                                int num_blocks, float scale, pa_dtype dtype, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, pa_stream_t stream);

/*
 * Whole-block copies between KV pools ([kwkr] §1.3 swap space; §2.2: the
 * block manager moves inactive physical blocks to host memory and back;
 * §1.3: physical blocks shared by several requests).  For each pair i,
 * (src, dst) = (pairs[2i], pairs[2i+1]): block src of the source pools is
 * copied byte for byte to block dst of the destination pools, K and V.
 * One call covers:
 *  - fork / copy inside one pool (source and destination pools the same);
 *  - swap out / in between the device pool and a host pool, whose memory
 *    must be reachable from the device (cudaHostAlloc / cudaHostRegister);
 *  - pack / unpack a request's blocks to / from a contiguous buffer (a pool
 *    whose blocks are numbered 0 .. n-1).
 *  block_bytes  bytes of one block of one pool: block_size*num_kv_heads*head_dim*elem
 *  pairs        device int32 [num_pairs][2]; a negative entry skips the pair;
 *               an entry past its pool's block count sets PA_ERR_OUT_OF_RANGE
 *               in *dev_status and the pair is skipped
 * Precondition (not checked on the device): destinations are distinct and no
 * destination block is also a source in the same call.
 */
PA_API pa_status pa_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                                int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                                const int32_t *pairs, int num_pairs, int32_t *dev_status,
                                pa_stream_t stream);

/* Workspace bytes pa_varlen_prefill needs for these sizes. */
PA_API size_t pa_varlen_prefill_workspace_size(int num_seqs, int total_q, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks);

/*
 * Varlen paged prefill over one concatenated super-sequence ([iitog] model
 * runner: all sequences concatenated, masks and positions keep each on its
 * own tokens; chunked prefill over a cached prefix).  Sequence s owns query
 * rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1; with q_len = that count and
 * ctx = context_lens[s] (cached prefix plus the new tokens, already written
 * to the pools), query row i sits at position ctx - q_len + i and attends
 * causally to keys 0 .. ctx - q_len + i of its own sequence only:
 *     out[row][h] = sum_{j <= pos} softmax_j(scale * <q[row][h], K_s[j][g]>) V_s[j][g].
 * Sequences with q_len == 1 (decode rows of a mixed step) take the decode
 * kernels; the others take the prefill kernel.  q_len == 0 is allowed and
 * produces nothing.  max_q_len bounds every q_len (a larger one sets
 * PA_ERR_OUT_OF_RANGE and its rows are unspecified).
 *  out, q       device [total_q][num_heads][head_dim]
 *  cu_seqlens_q device int32 [num_seqs + 1]
 *  workspace    >= pa_varlen_prefill_workspace_size(...) bytes, 16-byte aligned
 */
PA_API pa_status pa_varlen_prefill(void *out, const void *q, const int32_t *cu_seqlens_q,
                            const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens,
                            int num_seqs, int total_q, int max_q_len, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int max_blocks,
                            int num_blocks, float scale, pa_dtype dtype, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, pa_stream_t stream);

/*
 * One mixed continuous-batching step in one call ([iitog] model runner: the
 * new tokens' K/V go into their cache slots, then attention over the
 * super-sequence): exactly pa_compute_slot_mapping(block_tables, seq_start,
 * cu_seqlens_q, total_q) -> slot_mapping, then pa_reshape_and_cache of key /
 * value through it, then pa_varlen_prefill (same arguments, same results).
 * The new tokens are the query tokens: token t of sequence s
 * (cu_seqlens_q[s] <= t < cu_seqlens_q[s+1]) sits at position
 * seq_start[s] + t - cu_seqlens_q[s], and context_lens[s] must count it.
 * On the fast path (bf16, head_dim 64/128, 16-byte aligned rows and
 * strides, decode and prefill kernels both applicable, max_q_len > 1) the
 * slot mapping and the cache write run beside the attention's plan launch,
 * saving two launches; otherwise the three calls run one after the other.
 *  key, value   device [total_q][num_kv_heads][head_dim], token strides given
 *  seq_start    device int32 [num_seqs]: tokens cached before this step
 *  slot_mapping device int64 [total_q], written
 *  workspace    >= pa_varlen_prefill_workspace_size(...) bytes, 16-byte aligned
 */
PA_API pa_status pa_varlen_step(void *out, const void *q, const void *key, const void *value,
                                int64_t key_stride_tok, int64_t value_stride_tok, void *k_cache,
                                void *v_cache, const int32_t *cu_seqlens_q,
                                const int32_t *block_tables, const int32_t *context_lens,
                                const int32_t *seq_start, int64_t *slot_mapping, int num_seqs,
                                int total_q, int max_q_len, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int max_blocks, int num_blocks,
                                float scale, pa_dtype dtype, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, pa_stream_t stream);

/*
 * Encode-only varlen paged attention: pa_varlen_prefill without the causal
 * mask.  Every query row of sequence s attends to all context_lens[s] keys of
 * s, and still to no other sequence's ("vLLMつかったら、ベクトル検索サーバーが
 * 高速化して安定性も向上した": an embedding / vector-search server only
 * encodes).  Same arguments, layouts, workspace (pa_varlen_prefill_workspace_size)
 * and error behaviour as pa_varlen_prefill.
 */
PA_API pa_status pa_varlen_encode(void *out, const void *q, const int32_t *cu_seqlens_q,
                                  const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *context_lens,
                                  int num_seqs, int total_q, int max_q_len, int num_heads,
                                  int num_kv_heads, int head_dim, int block_size, int max_blocks,
                                  int num_blocks, float scale, pa_dtype dtype, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, pa_stream_t stream);

/*
 * Host block manager (no GPU work): the physical block pool that produces the
 * block tables above.  [iitog] allocate_slots paragraph: a pool of free blocks;
 * a request that grows by n tokens gets ceil((cached + n) / block_size) minus
 * its current number of blocks, when the pool holds that many, and nothing
 * otherwise (the scheduler then preempts or skips it).  [kwkr] §2.2: a
 * finished request's blocks return to the pool at once; §1.3: blocks can be
 * referenced read-only by several tables, so a block returns to the pool
 * when its last reference is freed.  All calls lock an internal mutex.
 */
typedef struct pa_block_manager pa_block_manager;

/* Pool of num_blocks blocks of block_size tokens; NULL on bad arguments. */
PA_API pa_block_manager *pa_block_manager_create(int num_blocks, int block_size,
                                                 int max_blocks_per_seq);
PA_API void pa_block_manager_destroy(pa_block_manager *m);
/* Free blocks in the pool, or -1 for a NULL manager. */
PA_API int pa_block_manager_num_free(pa_block_manager *m);
/* References to `block` (0 = free), or -1 when out of range. */
PA_API int pa_block_manager_refcount(pa_block_manager *m, int block);
/*
 * allocate_slots: room for num_new_tokens more tokens of seq_id (created on
 * first use).  PA_OK; PA_ERR_OUT_OF_RANGE when the pool lacks the blocks
 * (nothing is taken); PA_ERR_INVALID_ARG past max_blocks_per_seq;
 * PA_ERR_UNSUPPORTED when the last block is partly filled and shared (a write
 * into a shared block would need copy-on-write, which is not provided).
 */
PA_API pa_status pa_allocate_slots(pa_block_manager *m, int64_t seq_id, int num_new_tokens);
/*
 * allocate_slots for n sequences in one call, in order, under one lock (a
 * decode step grows every running sequence by a token).  statuses[i]
 * (nullable) receives what pa_allocate_slots(m, seq_ids[i],
 * num_new_tokens[i]) returns.  Returns PA_OK when all succeed, else the
 * first failure's status; PA_ERR_INVALID_ARG for a NULL manager or arrays.
 */
PA_API pa_status pa_allocate_slots_batch(pa_block_manager *m, const int64_t *seq_ids,
                                         const int32_t *num_new_tokens, int n, int32_t *statuses);
/* Drops seq_id's references; blocks no table references go back to the pool. */
PA_API pa_status pa_free_sequence(pa_block_manager *m, int64_t seq_id);
/*
 * child_id (new) references the first num_tokens tokens of parent_id, which
 * must be whole blocks (PA_ERR_UNSUPPORTED otherwise): a shared read-only
 * prefix such as a common system prompt, or a fork for parallel sampling.
 */
PA_API pa_status pa_share_prefix(pa_block_manager *m, int64_t parent_id, int64_t child_id,
                                 int num_tokens);
/*
 * Host int32 block_tables [n][max_blocks] (unused entries -1) and num_tokens
 * [n] of the listed sequences, ready to copy to the device.
 */
PA_API pa_status pa_block_manager_tables(pa_block_manager *m, const int64_t *seq_ids, int n,
                                         int32_t *block_tables, int max_blocks,
                                         int32_t *num_tokens);

/*
 * Host-side check of the preconditions the kernels rely on but do not test,
 * for tests and debug runs.  All pointers are HOST memory; nothing touches
 * the device.  [kwkr] §1.2-1.3: a sequence reaches its blocks through its
 * block table, block i of a sequence holding its tokens i*B..i*B+B-1, and
 * blocks may be referenced read-only by several tables (a shared prefix).
 *  block_tables  int32 [num_seqs][max_blocks]; only the first
 *                ceil(context_lens[s] / block_size) entries of row s are used
 *  context_lens  int32 [num_seqs], or NULL to skip checks 1-2 and 5
 *  slot_mapping  int64 [num_slots] (the slots a write will fill), or NULL
 * Checks, in this order (the first failure is reported):
 *   1 every context_lens[s] is in [1, max_blocks * block_size];
 *   2 every used table entry is in [0, num_blocks);
 *   3 every slot is < num_blocks * block_size (negative slots are padding);
 *   4 no slot appears twice;
 *   5 no slot lies in a block that two or more used table entries reference
 *     (a shared block is read-only; writing it needs copy-on-write).
 * Returns PA_OK; PA_ERR_OUT_OF_RANGE for checks 1-3; PA_ERR_INVALID_ARG for
 * checks 4-5 or bad sizes.  *failed_check (1-5, 0 when OK) and *bad_index
 * (the offending row of context_lens or block_tables, or the index into
 * slot_mapping) are set when non-NULL.
 */
PA_API pa_status pa_validate_inputs(const int32_t *block_tables, int num_seqs, int max_blocks,
                                    const int32_t *context_lens, const int64_t *slot_mapping,
                                    int num_slots, int block_size, int num_blocks,
                                    int *failed_check, int64_t *bad_index);

/*
 * Copies the device status word to *host_out after synchronising `stream`.
 * Returns PA_ERR_CUDA if the copy fails (for example after a sticky fault).
 */
PA_API pa_status pa_get_device_status(const int32_t *dev_status, int32_t *host_out, pa_stream_t stream);

/* Sets the device status word to PA_OK (asynchronous on `stream`). */
PA_API pa_status pa_reset_device_status(int32_t *dev_status, pa_stream_t stream);

/*
 * Optional timing hook for profiling (no counterpart on the pages).  When
 * both are non-NULL, ev_begin and ev_end (cudaEvent_t handles created by the
 * caller) are recorded on the call's stream immediately before and after the
 * main attention kernel of every later pa_decode / pa_varlen_prefill call made
 * from the same host thread, so that kernel can be timed on its own.  Pass
 * NULL, NULL to stop.  The events are not owned by the library.
 */
PA_API pa_status pa_set_timing_events(void *ev_begin, void *ev_end);

/*
 * Test hook for the bounded in-kernel waits (no counterpart on the pages).
 * Every wait inside the library's pipelined kernels gives up after a time
 * limit, records PA_ERR_TIMEOUT in *dev_status and lets its kernel return, so
 * a stuck pipeline never hangs the GPU.  This hook lets a test reach those
 * branches on purpose, without any fault: for every later pa_decode,
 * pa_decode_step, pa_varlen_prefill, pa_varlen_step and pa_varlen_encode call
 * made from the same host thread,
 *  limit_ns  bounds each wait (0: the default of one second);
 *  stall     makes one role of each CTA stop early and never give the signal
 *            the others wait for (nobody ever sets it, so their waits run out):
 *    PA_STALL_NONE      normal operation;
 *    PA_STALL_PRODUCER  the CTA's copy producer issues `after` copies (decode:
 *                       `after` blocks; prefill: `after` K/V tiles of keys or
 *                       values) and then stops, so the consumers wait for
 *                       data that never comes;
 *    PA_STALL_CONSUMER  the CTA's consumers (decode: the attention warps, after
 *                       `after` blocks; prefill: the MMA issuer, after `after`
 *                       K/V tiles) stop, so the producer waits for ring slots
 *                       that are never freed;
 *  sites     (device int32, nullable) receives, OR-ed, one PA_WAIT_* bit per
 *            role whose wait ran out (a role that stopped on purpose sets none).
 * A CTA's own copies in flight are always waited for (one-second limit)
 * before it exits.  The hook changes results only in that the stalled calls
 * time out; PA_STALL_NONE with limit 0 restores normal operation.  Returns
 * PA_ERR_INVALID_ARG for an unknown mode or a negative `after`.
 */
enum {
    PA_STALL_NONE = 0, PA_STALL_PRODUCER = 1, PA_STALL_CONSUMER = 2
};
enum {
    PA_WAIT_DECODE_PRODUCER = 1, PA_WAIT_DECODE_CONSUMER = 2, PA_WAIT_PREFILL_PRODUCER = 4,
    PA_WAIT_PREFILL_MMA = 8, PA_WAIT_PREFILL_SOFTMAX = 16
};
PA_API pa_status pa_set_wait_test(uint64_t limit_ns, int stall, int after, int32_t *sites);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
