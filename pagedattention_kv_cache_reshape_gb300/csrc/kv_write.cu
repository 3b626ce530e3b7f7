// kv_write.cu -- slot mapping and the KV-cache write ("reshape_and_cache").
//
// Slot mapping follows "vLLM изнутри: как устроен движок для быстрого
// инференса LLM" (model-runner paragraph: the slot map is built while inputs
// are prepared) and "vLLM：颠覆大模型推理的高效API服务引擎深度解析" §1.2-1.3
// (block table from logical to physical blocks of 16 tokens).  The write
// follows the same page's §1.3: the new token's K/V vectors are stored into
// its physical block.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// One thread per new token.  The owning sequence is found by binary search
// over cu_seqlens_q (non-decreasing, cu[0] = 0, cu[num_seqs] = total_new),
// staged in shared memory with one coalesced load when it fits (`staged`).
__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_tables, int num_seqs,
                                    int max_blocks, const int32_t *__restrict__ seq_start,
                                    const int32_t *__restrict__ cu_seqlens_q, int total_new,
                                    int block_size, int num_blocks,
                                    int64_t *__restrict__ slot_mapping, int32_t *status, int staged) {
    extern __shared__ int32_t cu_s[];
    grid_dependency_wait();      // inputs may come from the previous kernel
    grid_dependents_launch();
    const int32_t *cu = cu_seqlens_q;
    if (staged) {
        for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) cu_s[i] = __ldg(cu_seqlens_q + i);
        __syncthreads();
        cu = cu_s;
    }
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total_new) return;
    int lo = 0, hi = num_seqs;  // find the last s with cu[s] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int64_t pos = (int64_t)__ldg(seq_start + s) + (t - cu[s]);
    const int64_t logical = pos / block_size;
    int64_t slot = -1;
    if (pos < 0 || logical >= max_blocks) {
        set_status(status, PA_ERR_OUT_OF_RANGE);
    } else {
        const int32_t phys = __ldg(block_tables + (int64_t)s * max_blocks + logical);
        if (phys < 0 || phys >= num_blocks) set_status(status, PA_ERR_OUT_OF_RANGE);
        else slot = (int64_t)phys * block_size + (pos - logical * block_size);
    }
    slot_mapping[t] = slot;
}

// One warp per token: the token's [num_kv_heads * head_dim] row is one
// contiguous pool row, copied with VEC-byte vectors.
template <typename V>
__global__ void reshape_and_cache_kernel(const char *__restrict__ key,
                                         const char *__restrict__ value, int64_t key_stride_b,
                                         int64_t value_stride_b, char *__restrict__ k_cache,
                                         char *__restrict__ v_cache,
                                         const int64_t *__restrict__ slot_mapping,
                                         int num_tokens, int row_vecs, int64_t pool_slots,
                                         int32_t *status) {
    grid_dependency_wait();      // the slot mapping may come from the previous kernel
    grid_dependents_launch();
    const int warps = blockDim.x >> 5;
    const int t = blockIdx.x * warps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) return;  // padding token
    if (slot >= pool_slots) {
        if (lane == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const V *ks = reinterpret_cast<const V *>(key + t * key_stride_b);
    const V *vs = reinterpret_cast<const V *>(value + t * value_stride_b);
    V *kd = reinterpret_cast<V *>(k_cache) + slot * row_vecs;
    V *vd = reinterpret_cast<V *>(v_cache) + slot * row_vecs;
    // four vectors of K and of V per lane in flight before their stores
    constexpr int kBatch = 4;
    for (int i0 = lane; i0 < row_vecs; i0 += 32 * kBatch) {
        V kv[kBatch], vv[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + 32 * u;
            if (i < row_vecs) {
                kv[u] = __ldg(ks + i);
                vv[u] = __ldg(vs + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + 32 * u;
            if (i < row_vecs) {
                kd[i] = kv[u];
                vd[i] = vv[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t *block_tables, int num_seqs, int max_blocks,
                                const int32_t *seq_start, const int32_t *cu_seqlens_q,
                                int total_new, int block_size, int num_blocks,
                                int64_t *slot_mapping, int32_t *status, cudaStream_t stream) {
    if (total_new == 0) return cudaSuccess;
    const int threads = 256;
    const int grid = (total_new + threads - 1) / threads;
    const size_t cu_bytes = sizeof(int32_t) * ((size_t)num_seqs + 1);
    const int staged = cu_bytes <= 32 * 1024 ? 1 : 0;
    return launch_dependent(slot_mapping_kernel, dim3(grid), dim3(threads), staged ? cu_bytes : 0,
                            stream, block_tables, num_seqs, max_blocks, seq_start, cu_seqlens_q,
                            total_new, block_size, num_blocks, slot_mapping, status, staged);
}

cudaError_t launch_reshape_and_cache(const void *key, const void *value, int64_t key_stride,
                                     int64_t value_stride, void *k_cache, void *v_cache,
                                     const int64_t *slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int num_blocks, int elem_bytes, int32_t *status,
                                     cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elem_bytes;
    const int64_t ks = key_stride * elem_bytes, vs = value_stride * elem_bytes;
    auto aligned = [](const void *p, int64_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    const bool v16 = row_bytes % 16 == 0 && ks % 16 == 0 && vs % 16 == 0 && aligned(key, 16) &&
                     aligned(value, 16) && aligned(k_cache, 16) && aligned(v_cache, 16);
    const int threads = 256, warps = threads / 32;
    const int grid = (num_tokens + warps - 1) / warps;
    const int64_t pool_slots = (int64_t)num_blocks * block_size;
    const char *kp = static_cast<const char *>(key), *vp = static_cast<const char *>(value);
    char *kc = static_cast<char *>(k_cache), *vc = static_cast<char *>(v_cache);
    if (v16)
        return launch_dependent(reshape_and_cache_kernel<uint4>, dim3(grid), dim3(threads), 0, stream,
                                kp, vp, ks, vs, kc, vc, slot_mapping, num_tokens, (int)(row_bytes / 16),
                                pool_slots, status);
    // element-sized copies (rows are whole elements: 2 or 4 bytes)
    if (elem_bytes == 4)
        return launch_dependent(reshape_and_cache_kernel<uint32_t>, dim3(grid), dim3(threads), 0, stream,
                                kp, vp, ks, vs, kc, vc, slot_mapping, num_tokens, (int)(row_bytes / 4),
                                pool_slots, status);
    return launch_dependent(reshape_and_cache_kernel<uint16_t>, dim3(grid), dim3(threads), 0, stream,
                            kp, vp, ks, vs, kc, vc, slot_mapping, num_tokens, (int)(row_bytes / 2),
                            pool_slots, status);
}

}  // namespace pa
