// pa_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <functional>
#include <utility>

#include "pa.h"
#include "prefill_plan.cuh"

namespace pa {

// Paged-attention problem as seen by the launchers (all pointers on device).
struct AttnArgs {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *cu_seqlens_q;  // nullptr: one query row per sequence (decode)
    int num_seqs;
    int total_q;
    int max_q_len;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    int max_blocks;
    int num_blocks;
    float scale;
    pa_dtype dtype;
    int32_t *status;
    int causal = 1;  // 0: every query row sees all context_lens[s] keys (encode-only)
};

constexpr int kMaxPersistentCtas = 1024;

int device_sm_count();  // SM count of the current device (cached per device)

// cuTensorMapEncodeTiled from the driver, found through the runtime (the
// library does not link libcuda); nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Timing hook (pa_set_timing_events): records the caller's events, if set,
// around the main attention kernel.
void timing_begin(cudaStream_t stream);
void timing_end(cudaStream_t stream);

// Bounded-wait test settings (pa_set_wait_test) of the calling host thread,
// passed to the pipelined kernels as launch parameters.
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // default limit of an in-kernel wait
struct WaitTest {
    uint64_t limit_ns = kWaitLimitNs;
    int stall = PA_STALL_NONE;
    int after = 0;
    int32_t *sites = nullptr;
};
const WaitTest &wait_test();

cudaError_t launch_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                                const int32_t *seq_start, const int32_t *cu_seqlens_q,
                                int total_new, int block_size, int num_blocks,
                                int64_t *slot_mapping, int32_t *status, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t key_stride,
                                     int64_t value_stride, void *k_cache, void *v_cache,
                                     const int64_t *slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int num_blocks, int elem_bytes, int32_t *status,
                                     cudaStream_t stream);

// Whole-block copies between pools (device or device-accessible host memory).
cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                               const int32_t *pairs, int num_pairs, int32_t *status,
                               cudaStream_t stream);

// CUDA-core attention for every supported shape and dtype (one CTA per query
// row and kv-head).  row_filter selects the sequences it computes.
constexpr int kAllRows = 0, kSkipSingleRows = 1, kOnlySingleRows = 2;
cudaError_t launch_generic_attention(const AttnArgs &a, int row_filter, cudaStream_t stream);

// pa_decode's host-side argument checks, in pa_decode's order and with its
// status codes.  On PA_OK, *need is the workspace the call takes: the split
// decode's scratch, or 0 when it runs the CUDA-core kernel (no scratch) or
// num_seqs is 0.
pa_status decode_requirements(const void *out, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                              int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int max_blocks, int num_blocks, float scale, pa_dtype dtype, size_t *need);

// Persistent TMA + tensor-core split-KV decode (bf16, head_dim 64/128).
bool split_decode_supported(const AttnArgs &a);
size_t split_decode_workspace(int num_seqs, int num_heads, int head_dim, int max_blocks, int block_size);
// Cache write folded into the decode plan kernel (bf16 rows of 16-byte
// multiples, 16-byte aligned pointers and strides).
struct KvWriteArgs {
    const void *key;
    const void *value;
    int64_t key_stride_tok;     // elements
    int64_t value_stride_tok;
    const int32_t *seq_start;
    const int32_t *cu_seqlens_new;
    int total_new;
    int64_t *slot_mapping;
};

// With a.cu_seqlens_q set, only sequences with q_len == 1 are processed and
// their query/output row is cu_seqlens_q[s].  With `write`, the step's cache
// write runs in the plan kernel, before any cache read of the decode kernel.
// With `prefill` (a batch that also has prefill chunks), one extra CTA of the
// plan launch builds the prefill kernel's work list, the decode kernel keeps
// only the SMs its share of the work needs, and `between` launches the
// prefill kernel right behind the decode kernel, so it runs on the SMs the
// decode kernel leaves.
cudaError_t launch_split_decode(const AttnArgs &a, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream, bool timed, const KvWriteArgs *write = nullptr,
                                const PrefillPlanJob *prefill = nullptr,
                                const std::function<cudaError_t()> *between = nullptr);

// tcgen05 causal prefill for sequences with q_len >= 2 (bf16, head_dim 64/128,
// q-heads per kv-head a power of two up to 16).
bool prefill_tc_supported(const AttnArgs &a);
size_t prefill_workspace(int num_seqs, int total_q);
// The work list for the prefill kernel in `workspace`.
PrefillPlanJob prefill_plan_job(const AttnArgs &a, void *workspace);
// planned: the work list was built by the decode plan launch and this kernel
// runs behind the decode kernel of the same batch (see launch_split_decode).
cudaError_t launch_prefill_tc(const AttnArgs &a, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream, bool planned = false);

// Launch as a programmatic dependent of the previous kernel in the stream:
// the kernel calls griddepcontrol.wait before it reads that kernel's output.
template <typename... KArgs, typename... Args>
inline
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pa
