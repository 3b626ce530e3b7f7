// pa_api.cu -- the extern "C" entry points declared in include/pa.h: host-side
// argument validation, workspace sizing and dispatch to the kernels.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

int device_sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
thread_local cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;
thread_local WaitTest g_wait_test;

}  // namespace

const WaitTest &wait_test() { return g_wait_test; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

void timing_begin(cudaStream_t stream) {
    if (g_ev_begin && g_ev_end) cudaEventRecord(g_ev_begin, stream);
}
void timing_end(cudaStream_t stream) {
    if (g_ev_begin && g_ev_end) cudaEventRecord(g_ev_end, stream);
}

namespace {

pa_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return PA_ERR_CUDA;
}

int elem_bytes(pa_dtype d) {
    return d == PA_DTYPE_F32 ? 4 : (d == PA_DTYPE_BF16 ? 2 : 0);
}

bool aligned(const void *p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// Shape checks shared by the attention calls.
pa_status check_attention_shape(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks, int num_blocks, pa_dtype dtype,
                                float scale) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;  // NaN
    if (elem_bytes(dtype) == 0) return PA_ERR_INVALID_ARG;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 32) return PA_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks * block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

}  // namespace

pa_status decode_requirements(const void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks, int num_blocks, float scale, pa_dtype dtype, size_t *need) {
    *need = 0;
    pa_status st = check_attention_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                         max_blocks, num_blocks, dtype, scale);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    if (!aligned(out, eb) || !aligned(q, eb) || !aligned(k_cache, eb) || !aligned(v_cache, eb))
        return PA_ERR_INVALID_ARG;
    AttnArgs a{const_cast<void *>(out), q, k_cache, v_cache, block_tables, context_lens, nullptr,
               num_seqs, num_seqs, 1, num_heads, num_kv_heads, head_dim, block_size,
               max_blocks, num_blocks, scale, dtype, nullptr};
    if (split_decode_supported(a))
        *need = split_decode_workspace(num_seqs, num_heads, head_dim, max_blocks, block_size);
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_version(void) { return 100; }

int pa_num_blocks_needed(int num_tokens, int block_size) {
    if (num_tokens < 0 || block_size <= 0) return -1;
    return num_tokens / block_size + (num_tokens % block_size != 0 ? 1 : 0);
}

pa_status pa_compute_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                                  const int32_t *seq_start, const int32_t *cu_seqlens_q,
                                  int total_new, int block_size, int num_blocks,
                                  int64_t *slot_mapping, int32_t *dev_status,
                                  pa_stream_t stream) {
    if (num_seqs < 0 || total_new < 0 || max_blocks <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (total_new > 0 && num_seqs == 0) return PA_ERR_INVALID_ARG;
    if (total_new == 0) return PA_OK;
    if (!block_tables || !seq_start || !cu_seqlens_q || !slot_mapping) return PA_ERR_INVALID_ARG;
    return from_cuda(launch_slot_mapping(block_tables, num_seqs, max_blocks, seq_start,
                                         cu_seqlens_q, total_new, block_size, num_blocks,
                                         slot_mapping, dev_status, (cudaStream_t)stream));
}

pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t key_stride_tok,
                               int64_t value_stride_tok, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                               int32_t *dev_status, pa_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0 || num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (key_stride_tok < row || value_stride_tok < row) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned(key, eb) || !aligned(value, eb) || !aligned(k_cache, eb) || !aligned(v_cache, eb))
        return PA_ERR_INVALID_ARG;
    return from_cuda(launch_reshape_and_cache(key, value, key_stride_tok, value_stride_tok,
                                              k_cache, v_cache, slot_mapping, num_tokens,
                                              num_kv_heads, head_dim, block_size, num_blocks, eb,
                                              dev_status, (cudaStream_t)stream));
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks) {
    (void)num_kv_heads;
    if (num_seqs < 0) num_seqs = 0;
    if (num_heads < 1) num_heads = 1;
    if (head_dim < 1) head_dim = 1;
    if (max_blocks < 1) max_blocks = 1;
    if (block_size < 1) block_size = 1;
    return split_decode_workspace(num_seqs, num_heads, head_dim, max_blocks, block_size);
}

pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                    int num_heads, int num_kv_heads, int head_dim, int block_size,
                    int max_blocks, int num_blocks, float scale, pa_dtype dtype,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status,
                    pa_stream_t stream) {
    size_t need = 0;
    const pa_status st = decode_requirements(out, q, k_cache, v_cache, block_tables, context_lens,
                                             num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                             max_blocks, num_blocks, scale, dtype, &need);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    AttnArgs a{out, q, k_cache, v_cache, block_tables, context_lens, nullptr,
               num_seqs, num_seqs, 1, num_heads, num_kv_heads, head_dim, block_size,
               max_blocks, num_blocks, scale, dtype, dev_status};
    cudaStream_t s = (cudaStream_t)stream;
    if (need > 0) {
        if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
        return from_cuda(launch_split_decode(a, workspace, workspace_bytes, s, true));
    }
    timing_begin(s);
    const cudaError_t e = launch_generic_attention(a, kAllRows, s);
    timing_end(s);
    return from_cuda(e);
}

pa_status pa_decode_step(void *out, const void *q, const void *key, const void *value,
                         int64_t key_stride_tok, int64_t value_stride_tok, void *k_cache,
                         void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                         const int32_t *seq_start, const int32_t *cu_seqlens_new, int total_new,
                         int64_t *slot_mapping, int num_seqs, int num_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks, int num_blocks, float scale,
                         pa_dtype dtype, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, pa_stream_t stream) {
    pa_status st = check_attention_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                         max_blocks, num_blocks, dtype, scale);
    if (st != PA_OK) return st;
    if (total_new < 0) return PA_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (total_new > 0) {
        if (num_seqs == 0 || !key || !value || !seq_start || !cu_seqlens_new || !slot_mapping)
            return PA_ERR_INVALID_ARG;
        if (key_stride_tok < row || value_stride_tok < row) return PA_ERR_INVALID_ARG;
    }
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned(out, eb) || !aligned(q, eb) || !aligned(k_cache, eb) || !aligned(v_cache, eb))
        return PA_ERR_INVALID_ARG;
    AttnArgs a{out, q, k_cache, v_cache, block_tables, context_lens, nullptr,
               num_seqs, num_seqs, 1, num_heads, num_kv_heads, head_dim, block_size,
               max_blocks, num_blocks, scale, dtype, dev_status};
    const bool fused = split_decode_supported(a) && total_new > 0 && aligned(key, 16) &&
                       aligned(value, 16) && (key_stride_tok * eb) % 16 == 0 &&
                       (value_stride_tok * eb) % 16 == 0 && (row * eb) % 16 == 0;
    if (!fused) {
        if (total_new > 0) {
            st = pa_compute_slot_mapping(block_tables, num_seqs, max_blocks, seq_start, cu_seqlens_new,
                                         total_new, block_size, num_blocks, slot_mapping, dev_status, stream);
            if (st != PA_OK) return st;
            st = pa_reshape_and_cache(key, value, key_stride_tok, value_stride_tok, k_cache, v_cache,
                                      slot_mapping, total_new, num_kv_heads, head_dim, block_size,
                                      num_blocks, dtype, dev_status, stream);
            if (st != PA_OK) return st;
        }
        return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                         num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale, dtype,
                         workspace, workspace_bytes, dev_status, stream);
    }
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 block_size, max_blocks);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
    KvWriteArgs wr{key, value, key_stride_tok, value_stride_tok, seq_start, cu_seqlens_new,
                   total_new, slot_mapping};
    return from_cuda(launch_split_decode(a, workspace, workspace_bytes, (cudaStream_t)stream, true, &wr));
}

pa_status pa_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                         int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                         const int32_t *pairs, int num_pairs, int32_t *dev_status,
                         pa_stream_t stream) {
    if (num_pairs < 0 || block_bytes <= 0 || src_num_blocks < 0 || dst_num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if (block_bytes % 2 != 0) return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !pairs) return PA_ERR_INVALID_ARG;
    if (!aligned(src_k, 2) || !aligned(src_v, 2) || !aligned(dst_k, 2) || !aligned(dst_v, 2))
        return PA_ERR_INVALID_ARG;
    return from_cuda(launch_copy_blocks(src_k, src_v, dst_k, dst_v, block_bytes, src_num_blocks,
                                        dst_num_blocks, pairs, num_pairs, dev_status,
                                        (cudaStream_t)stream));
}

size_t pa_varlen_prefill_workspace_size(int num_seqs, int total_q, int num_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int max_blocks) {
    if (total_q < 0) total_q = 0;
    if (num_seqs < 0) num_seqs = 0;
    return pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                    max_blocks) +
           prefill_workspace(num_seqs, total_q);
}

}  // extern "C"

namespace {
pa_status varlen_attention(void *out, const void *q, const int32_t *cu_seqlens_q,
                           const void *k_cache, const void *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int num_seqs, int total_q, int max_q_len,
                           int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks, int num_blocks, float scale, pa_dtype dtype,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           pa_stream_t stream, int causal, const KvWriteArgs *write = nullptr) {
    pa_status st = check_attention_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                         max_blocks, num_blocks, dtype, scale);
    if (st != PA_OK) return st;
    if (total_q < 0 || max_q_len < 0) return PA_ERR_INVALID_ARG;
    if (total_q == 0 || num_seqs == 0) return PA_OK;
    if (!out || !q || !cu_seqlens_q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    const int eb = elem_bytes(dtype);
    if (!aligned(out, eb) || !aligned(q, eb) || !aligned(k_cache, eb) || !aligned(v_cache, eb))
        return PA_ERR_INVALID_ARG;
    AttnArgs a{out, q, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q,
               num_seqs, total_q, max_q_len, num_heads, num_kv_heads, head_dim, block_size,
               max_blocks, num_blocks, scale, dtype, dev_status, causal};
    cudaStream_t s = (cudaStream_t)stream;
    const bool fast_decode = split_decode_supported(a);
    const bool fast_prefill = prefill_tc_supported(a);
    const size_t dec_ws = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                   block_size, max_blocks);
    if (fast_decode || fast_prefill) {
        const size_t need = pa_varlen_prefill_workspace_size(num_seqs, total_q, num_heads,
                                                             num_kv_heads, head_dim, block_size,
                                                             max_blocks);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 16)) return PA_ERR_WORKSPACE;
    }
    // the step's cache write (pa_varlen_step): beside the plan launch of the
    // shared chain when its rows are 16-byte vectors, else ahead of attention
    const bool fold_write = write && fast_decode && fast_prefill && max_q_len > 1 &&
                            aligned(write->key, 16) && aligned(write->value, 16) &&
                            (write->key_stride_tok * eb) % 16 == 0 && (write->value_stride_tok * eb) % 16 == 0 &&
                            ((int64_t)num_kv_heads * head_dim * eb) % 16 == 0;
    if (write && !fold_write) {
        st = pa_compute_slot_mapping(block_tables, num_seqs, max_blocks, write->seq_start,
                                     write->cu_seqlens_new, write->total_new, block_size, num_blocks,
                                     write->slot_mapping, dev_status, stream);
        if (st != PA_OK) return st;
        st = pa_reshape_and_cache(write->key, write->value, write->key_stride_tok, write->value_stride_tok,
                                  const_cast<void *>(k_cache), const_cast<void *>(v_cache), write->slot_mapping,
                                  write->total_new, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                                  dev_status, stream);
        if (st != PA_OK) return st;
    }
    // decode rows (q_len == 1) stream through the split-KV decode kernels,
    // prefill chunks (q_len >= 2) through the tensor-core prefill kernel
    timing_begin(s);
    cudaError_t e = cudaSuccess;
    if (fast_decode && fast_prefill && max_q_len > 1) {
        // both parts in one chain on this stream: one plan launch for both,
        // the decode kernel (it keeps the SMs its share of the work needs and
        // frees the rest at once), the persistent prefill kernel as its
        // programmatic dependent (it starts only when every decode CTA is
        // resident, then takes each SM the decode kernel frees)
        uint8_t *pws = static_cast<uint8_t *>(workspace) + dec_ws;
        const PrefillPlanJob job = prefill_plan_job(a, pws);
        const std::function<cudaError_t()> prefill = [&]() {
            return launch_prefill_tc(a, pws, workspace_bytes - dec_ws, s, true);
        };
        e = launch_split_decode(a, workspace, dec_ws, s, false, fold_write ? write : nullptr, &job, &prefill);
        timing_end(s);
        return from_cuda(e);
    }
    if (fast_decode) {
        e = launch_split_decode(a, workspace, dec_ws, s, false);
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (max_q_len > 1 || !fast_decode) {
        if (fast_prefill && max_q_len > 1) {
            e = launch_prefill_tc(a, static_cast<uint8_t *>(workspace) + dec_ws, workspace_bytes - dec_ws, s);
            if (e == cudaSuccess && !fast_decode) e = launch_generic_attention(a, kOnlySingleRows, s);
        } else {
            e = launch_generic_attention(a, fast_decode ? kSkipSingleRows : kAllRows, s);
        }
    }
    timing_end(s);
    return from_cuda(e);
}
}  // namespace

extern "C" {

pa_status pa_varlen_prefill(void *out, const void *q, const int32_t *cu_seqlens_q,
                            const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens,
                            int num_seqs, int total_q, int max_q_len, int num_heads,
                            int num_kv_heads, int head_dim, int block_size, int max_blocks,
                            int num_blocks, float scale, pa_dtype dtype, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status, pa_stream_t stream) {
    return varlen_attention(out, q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens,
                            num_seqs, total_q, max_q_len, num_heads, num_kv_heads, head_dim,
                            block_size, max_blocks, num_blocks, scale, dtype, workspace,
                            workspace_bytes, dev_status, stream, 1);
}

pa_status pa_varlen_encode(void *out, const void *q, const int32_t *cu_seqlens_q,
                           const void *k_cache, const void *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int num_seqs, int total_q, int max_q_len,
                           int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_blocks, int num_blocks, float scale, pa_dtype dtype,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           pa_stream_t stream) {
    return varlen_attention(out, q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens,
                            num_seqs, total_q, max_q_len, num_heads, num_kv_heads, head_dim,
                            block_size, max_blocks, num_blocks, scale, dtype, workspace,
                            workspace_bytes, dev_status, stream, 0);
}

pa_status pa_varlen_step(void *out, const void *q, const void *key, const void *value,
                         int64_t key_stride_tok, int64_t value_stride_tok, void *k_cache, void *v_cache,
                         const int32_t *cu_seqlens_q, const int32_t *block_tables,
                         const int32_t *context_lens, const int32_t *seq_start, int64_t *slot_mapping,
                         int num_seqs, int total_q, int max_q_len, int num_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_blocks, int num_blocks, float scale,
                         pa_dtype dtype, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         pa_stream_t stream) {
    pa_status st = check_attention_shape(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                         max_blocks, num_blocks, dtype, scale);
    if (st != PA_OK) return st;
    if (total_q < 0 || max_q_len < 0) return PA_ERR_INVALID_ARG;
    if (total_q == 0 || num_seqs == 0) return PA_OK;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (!key || !value || !seq_start || !cu_seqlens_q || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (key_stride_tok < row || value_stride_tok < row) return PA_ERR_INVALID_ARG;
    const KvWriteArgs wr{key, value, key_stride_tok, value_stride_tok, seq_start, cu_seqlens_q,
                         total_q, slot_mapping};
    return varlen_attention(out, q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                            total_q, max_q_len, num_heads, num_kv_heads, head_dim, block_size, max_blocks,
                            num_blocks, scale, dtype, workspace, workspace_bytes, dev_status, stream, 1, &wr);
}

pa_status pa_get_device_status(const int32_t *dev_status, int32_t *host_out, pa_stream_t stream) {
    if (!dev_status || !host_out) return PA_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return from_cuda(e);
}

pa_status pa_reset_device_status(int32_t *dev_status, pa_stream_t stream) {
    if (!dev_status) return PA_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), (cudaStream_t)stream));
}

pa_status pa_set_timing_events(void *ev_begin, void *ev_end) {
    if ((ev_begin == nullptr) != (ev_end == nullptr)) return PA_ERR_INVALID_ARG;
    g_ev_begin = static_cast<cudaEvent_t>(ev_begin);
    g_ev_end = static_cast<cudaEvent_t>(ev_end);
    return PA_OK;
}

pa_status pa_set_wait_test(uint64_t limit_ns, int stall, int after, int32_t *sites) {
    if (stall < PA_STALL_NONE || stall > PA_STALL_CONSUMER || after < 0) return PA_ERR_INVALID_ARG;
    g_wait_test.limit_ns = limit_ns == 0 ? kWaitLimitNs : limit_ns;
    g_wait_test.stall = stall;
    g_wait_test.after = after;
    g_wait_test.sites = sites;
    return PA_OK;
}

}  // extern "C"
