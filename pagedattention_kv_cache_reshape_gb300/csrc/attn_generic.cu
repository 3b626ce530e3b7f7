// attn_generic.cu -- CUDA-core paged attention for every supported shape:
// fp32 or bf16, head_dim 64/128, any q-heads per kv-head up to 32, decode or
// causal varlen prefill.  One CTA per (query row, kv-head) walks the row's
// visible keys in tiles of 64 through the block table ("vLLM：颠覆大模型推理
// 的高效API服务引擎深度解析" §1.3: gather the scattered physical blocks into
// a logically contiguous KV), keeping a running max and sum per q-head
// (online softmax) with fp32 arithmetic throughout.
//
// It is the path for fp32 inputs and for shapes the tensor-core kernels do
// not cover, and the prefill path for bf16 until the tcgen05 kernel takes
// over.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 128;
constexpr int kMaxGroup = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    generic_attention_kernel(AttnArgs a, int row_filter) {
    extern __shared__ float smem[];
    const int G = a.num_heads / a.num_kv_heads;
    float *q_s = smem;                  // [G][D]
    float *o_s = q_s + G * D;           // [G][D]  output accumulators
    float *p_s = o_s + G * D;           // [G][kTile] logits, then weights
    float *m_s = p_s + G * kTile;       // [G] running max
    float *l_s = m_s + G;               // [G] running sum
    float *alpha_s = l_s + G;           // [G] rescale factor of this tile
    int *blk_s = reinterpret_cast<int *>(alpha_s + G);  // [kTile] physical block per key
    __shared__ int bad;

    const int row = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kThreads / 32;

    // ---- which sequence owns this query row
    int s, first, q_len;
    if (a.cu_seqlens_q) {
        int lo = 0, hi = a.num_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(a.cu_seqlens_q + mid) <= row) lo = mid; else hi = mid;
        }
        s = lo;
        first = __ldg(a.cu_seqlens_q + s);
        q_len = __ldg(a.cu_seqlens_q + s + 1) - first;
    } else {
        s = row;
        first = row;
        q_len = 1;
    }
    const int i = row - first;
    if ((row_filter == kSkipSingleRows && q_len == 1) || (row_filter == kOnlySingleRows && q_len != 1))
        return;
    const int ctx = __ldg(a.context_lens + s);
    if (i < 0 || i >= q_len || ctx <= 0 || (int64_t)ctx > (int64_t)a.max_blocks * a.block_size ||
        q_len > ctx || q_len > a.max_q_len) {
        if (tid == 0) set_status(a.status, PA_ERR_OUT_OF_RANGE);
        return;
    }
    // keys 0 .. position of this query (causal), or the whole sequence (encode)
    const int n_keys = a.causal ? ctx - q_len + i + 1 : ctx;

    const T *q = static_cast<const T *>(a.q) + ((int64_t)row * a.num_heads + g * G) * D;
    for (int idx = tid; idx < G * D; idx += kThreads) {
        q_s[idx] = to_float(q[idx]);
        o_s[idx] = 0.f;
    }
    if (tid < G) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    if (tid == 0) bad = 0;
    __syncthreads();

    const T *kc = static_cast<const T *>(a.k_cache);
    const T *vc = static_cast<const T *>(a.v_cache);
    const int32_t *bt = a.block_tables + (int64_t)s * a.max_blocks;
    const int B = a.block_size;
    const int64_t head_stride = D, tok_stride = (int64_t)a.num_kv_heads * D;

    for (int j0 = 0; j0 < n_keys; j0 += kTile) {
        const int jn = min(kTile, n_keys - j0);
        // ---- logits: warp w takes keys w, w+4, ...; lanes split head_dim
        for (int jj = warp; jj < jn; jj += kWarps) {
            const int j = j0 + jj;
            const int32_t blk = __ldg(bt + j / B);
            if (blk < 0 || blk >= a.num_blocks) {
                if (lane == 0) {
                    set_status(a.status, PA_ERR_OUT_OF_RANGE);
                    bad = 1;
                    blk_s[jj] = -1;
                }
                for (int h = lane; h < G; h += 32) p_s[h * kTile + jj] = -INFINITY;
                continue;
            }
            const T *krow = kc + ((int64_t)blk * B + (j % B)) * tok_stride + g * head_stride;
            float kv[D / 32];
#pragma unroll
            for (int t = 0; t < D / 32; ++t) kv[t] = to_float(krow[lane + 32 * t]);
            for (int h = 0; h < G; ++h) {
                float part = 0.f;
#pragma unroll
                for (int t = 0; t < D / 32; ++t) part = fmaf(q_s[h * D + lane + 32 * t], kv[t], part);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                if (lane == 0) p_s[h * kTile + jj] = part * a.scale;
            }
            if (lane == 0) blk_s[jj] = blk;
        }
        __syncthreads();
        // ---- online softmax update: warp w takes q-heads w, w+4, ...
        for (int h = warp; h < G; h += kWarps) {
            float tmax = -INFINITY;
            for (int jj = lane; jj < jn; jj += 32) tmax = fmaxf(tmax, p_s[h * kTile + jj]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_old = m_s[h];
            const float m_new = fmaxf(m_old, tmax);
            float alpha, sum = 0.f;
            if (m_new == -INFINITY) {
                alpha = 1.f;
                for (int jj = lane; jj < kTile; jj += 32) p_s[h * kTile + jj] = 0.f;
            } else {
                alpha = expf(m_old - m_new);
                for (int jj = lane; jj < kTile; jj += 32) {
                    const float p = jj < jn ? expf(p_s[h * kTile + jj] - m_new) : 0.f;
                    p_s[h * kTile + jj] = p;
                    sum += p;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) {
                l_s[h] = l_s[h] * alpha + sum;
                m_s[h] = m_new;
                alpha_s[h] = alpha;
            }
        }
        __syncthreads();
        // ---- P x V: thread d accumulates column d of every q-head
        if (tid < D) {
            float v[kTile];
#pragma unroll
            for (int jj = 0; jj < kTile; ++jj) {
                v[jj] = 0.f;
                if (jj < jn) {
                    const int blk = blk_s[jj];
                    if (blk >= 0) {
                        const int j = j0 + jj;
                        v[jj] = to_float(vc[((int64_t)blk * B + (j % B)) * tok_stride +
                                            g * head_stride + tid]);
                    }
                }
            }
            for (int h = 0; h < G; ++h) {
                float acc = o_s[h * D + tid] * alpha_s[h];
#pragma unroll
                for (int jj = 0; jj < kTile; ++jj) acc = fmaf(p_s[h * kTile + jj], v[jj], acc);
                o_s[h * D + tid] = acc;
            }
        }
        __syncthreads();
    }
    if (bad) return;
    T *out = static_cast<T *>(a.out) + ((int64_t)row * a.num_heads + g * G) * D;
    if (tid < D) {
        for (int h = 0; h < G; ++h) out[h * D + tid] = from_float<T>(o_s[h * D + tid] / l_s[h]);
    }
}

template <typename T, int D>
cudaError_t launch_typed(const AttnArgs &a, int row_filter, cudaStream_t stream) {
    const int G = a.num_heads / a.num_kv_heads;
    const size_t smem = sizeof(float) * (2 * G * D + G * kTile + 3 * G) + sizeof(int) * kTile;
    auto kern = generic_attention_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.total_q, a.num_kv_heads);
    kern<<<grid, kThreads, smem, stream>>>(a, row_filter);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic_attention(const AttnArgs &a, int row_filter, cudaStream_t stream) {
    if (a.total_q == 0 || a.num_seqs == 0) return cudaSuccess;
    if (a.num_heads / a.num_kv_heads > kMaxGroup) return cudaErrorInvalidValue;
    if (a.dtype == PA_DTYPE_F32) {
        return a.head_dim == 64 ? launch_typed<float, 64>(a, row_filter, stream)
                                : launch_typed<float, 128>(a, row_filter, stream);
    }
    return a.head_dim == 64 ? launch_typed<__nv_bfloat16, 64>(a, row_filter, stream)
                            : launch_typed<__nv_bfloat16, 128>(a, row_filter, stream);
}

}  // namespace pa
