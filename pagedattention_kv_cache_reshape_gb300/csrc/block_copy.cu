// block_copy.cu -- whole-block copies between KV pools: fork inside one pool,
// swap between the device pool and a pinned host pool, pack / unpack a
// request's blocks to / from a contiguous transfer buffer.
//
// "vLLM：颠覆大模型推理的高效API服务引擎深度解析" §1.3 (swap space) and §2.2
// (the block manager moves inactive physical blocks to host memory and back
// when device memory runs short); §1.3 (blocks shared by several requests).
// A block of one pool is one contiguous slab of block_size * num_kv_heads *
// head_dim elements, so every case is the same copy of (src, dst) slabs.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kVecsPerThread = 4;   // 16 KB of one block per CTA and pool

// grid: (pair, chunk of the block).  V is the copy unit (uint4 or narrower).
template <typename V>
__global__ void __launch_bounds__(kThreads)
    copy_blocks_kernel(const V *__restrict__ src_k, const V *__restrict__ src_v,
                       V *__restrict__ dst_k, V *__restrict__ dst_v, int64_t block_vecs,
                       int src_num_blocks, int dst_num_blocks, const int32_t *__restrict__ pairs,
                       int32_t *status) {
    grid_dependency_wait();
    grid_dependents_launch();
    const int i = blockIdx.x;
    const int32_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || dst < 0) return;
    if (src >= src_num_blocks || dst >= dst_num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int64_t base = (int64_t)blockIdx.y * kThreads * kVecsPerThread;
    const V *sk = src_k + src * block_vecs, *sv = src_v + src * block_vecs;
    V *dk = dst_k + dst * block_vecs, *dv = dst_v + dst * block_vecs;
    V kr[kVecsPerThread], vr[kVecsPerThread];
#pragma unroll
    for (int u = 0; u < kVecsPerThread; ++u) {
        const int64_t e = base + u * kThreads + threadIdx.x;
        if (e < block_vecs) {
            kr[u] = sk[e];
            vr[u] = sv[e];
        }
    }
#pragma unroll
    for (int u = 0; u < kVecsPerThread; ++u) {
        const int64_t e = base + u * kThreads + threadIdx.x;
        if (e < block_vecs) {
            dk[e] = kr[u];
            dv[e] = vr[u];
        }
    }
}

template <typename V>
cudaError_t launch_typed(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                         int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                         const int32_t *pairs, int num_pairs, int32_t *status, cudaStream_t stream) {
    const int64_t block_vecs = block_bytes / (int64_t)sizeof(V);
    const int64_t per_cta = (int64_t)kThreads * kVecsPerThread;
    const dim3 grid(num_pairs, (unsigned)((block_vecs + per_cta - 1) / per_cta));
    return launch_dependent(copy_blocks_kernel<V>, grid, dim3(kThreads), 0, stream,
                            static_cast<const V *>(src_k), static_cast<const V *>(src_v),
                            static_cast<V *>(dst_k), static_cast<V *>(dst_v), block_vecs,
                            src_num_blocks, dst_num_blocks, pairs, status);
}

}  // namespace

cudaError_t launch_copy_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                               const int32_t *pairs, int num_pairs, int32_t *status,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    auto al = [](const void *p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
    const bool v16 = block_bytes % 16 == 0 && al(src_k, 16) && al(src_v, 16) && al(dst_k, 16) && al(dst_v, 16);
    if (v16)
        return launch_typed<uint4>(src_k, src_v, dst_k, dst_v, block_bytes, src_num_blocks,
                                   dst_num_blocks, pairs, num_pairs, status, stream);
    return launch_typed<uint16_t>(src_k, src_v, dst_k, dst_v, block_bytes, src_num_blocks,
                                  dst_num_blocks, pairs, num_pairs, status, stream);
}

}  // namespace pa
