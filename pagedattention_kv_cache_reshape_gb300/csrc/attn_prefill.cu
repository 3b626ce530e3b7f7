// attn_prefill.cu -- causal varlen paged prefill on the 5th-gen tensor cores
// (tcgen05 MMA with TMEM accumulators, operands staged by TMA).
//
// What it computes ("vLLM изнутри…", model-runner paragraph: the batch is one
// concatenated super-sequence whose masks and positions keep every sequence
// on its own tokens; chunked prefill attends to its cached prefix plus
// itself; "vLLM：颠覆大模型推理的高效API服务引擎深度解析" §1.3: keys and
// values are gathered through the block table): for sequence s with q_len
// new tokens and ctx = context_lens[s], query row i (position
// ctx - q_len + i) and q-head h,
//     out[row][h] = sum_{j <= pos} softmax_j(scale * <q[row][h], K_s[j][g(h)]>) V_s[j][g(h)].
//
// Work unit (one CTA): 128 rows = POS consecutive query positions x the G
// query heads of one kv-head (so each K/V tile is loaded once for the whole
// group), against the sequence's keys in tiles of 64 (4 cache blocks); two
// CTAs share an SM so two softmax warpgroups overlap each other's MMAs.
// Warp roles: warps 0-3 softmax + epilogue (thread = row = TMEM lane),
// warp 4 TMA producer, warp 5 TMEM owner and MMA issuer (one thread).
//   S_j = Q K_j^T   -> TMEM (two buffers, so S_{j+1} overlaps softmax j)
//   P_j = exp2(S_j * scale*log2e - m)  (bf16, shared memory, K-major)
//   O  += P_j V_j   -> TMEM (fp32)
// The running max is only raised (and O rescaled in TMEM) when a row's max
// grows by more than 2^8; otherwise the stale max is kept, which changes no
// result because l uses the same max.  Causal masking is a select on the
// logits; keys of blocks past the sequence end come in as zeros (TMA
// out-of-bounds fill), and value rows past the context end inside the last
// block are zeroed in shared memory so P * V never sees 0 * NaN.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kB = kBlockSize;
constexpr int BM = 128;               // rows per tile
constexpr int BN = 64;                // keys per KV tile (4 cache blocks)
constexpr int kBlocksPerTile = BN / kB;
constexpr int kThreads = 192;
constexpr int kPlanThreads = 512;
constexpr int kTmemCols = 256;        // two CTAs share an SM's 512 columns
constexpr uint32_t kSColStride = BN;  // S buffer b at TMEM column b * BN
constexpr uint32_t kOCol = 2 * BN;    // O after the two S buffers

struct PrefillParams {
    const int32_t *cu_seqlens_q;
    const int32_t *context_lens;
    const int32_t *block_tables;
    const int2 *entries;       // (sequence, tile) per CTA
    const int32_t *num_entries;
    __nv_bfloat16 *out;
    int num_seqs;
    int total_q;
    int max_q_len;
    int num_heads;
    int group;       // q-heads per kv-head
    int pos_shift;   // log2(query positions per tile) = log2(128 / group)
    int max_blocks;
    int num_blocks;
    float scale_log2;
    int32_t *status;
};

// ------------------------------------------------------------------ plan
// One CTA: tiles per sequence with q_len >= 2, exclusive scan, one entry per
// tile (the tile with the most keys first inside each sequence).
__global__ void __launch_bounds__(kPlanThreads)
    prefill_plan_kernel(const int32_t *__restrict__ cu_seqlens_q, int num_seqs, int pos_shift,
                        int2 *__restrict__ entries, int32_t *__restrict__ count, int capacity) {
    __shared__ int warp_tot[kPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pos = 1 << pos_shift;
    int running = 0;
    for (int base = 0; base < num_seqs; base += kPlanThreads) {
        const int s = base + tid;
        int nt = 0;
        if (s < num_seqs) {
            const int ql = __ldg(cu_seqlens_q + s + 1) - __ldg(cu_seqlens_q + s);
            if (ql > 1) nt = (ql + pos - 1) >> pos_shift;
        }
        int incl = nt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int warp_off = 0, chunk_tot = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            if (w < warp) warp_off += warp_tot[w];
            chunk_tot += warp_tot[w];
        }
        const int first = running + warp_off + incl - nt;
        for (int t = 0; t < nt; ++t)
            if (first + t < capacity) entries[first + t] = make_int2(s, nt - 1 - t);
        running += chunk_tot;
        __syncthreads();
    }
    if (tid == 0) *count = running < capacity ? running : capacity;
}

// ------------------------------------------------------------------ main kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    constexpr int kDH = D / 64;             // 64-column planes of a head
    constexpr int kQBytes = BM * D * 2;
    constexpr int kKVBytes = BN * D * 2;    // K (or V) of one tile
    constexpr int kPlaneQ = BM * 128;       // one 64-column plane of Q or P
    constexpr int kPlaneKV = BN * 128;      // one 64-column plane of K or V
    constexpr uint32_t kIdescQK = umma_idesc_bf16(BM, BN, 0);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(BM, D, 1);

    // all shared state is dynamic (no static shared memory), so the 1024-byte
    // aligned operand tiles start at offset 0 and two CTAs fit on one SM
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *q_s = smem;
    uint8_t *k_s0 = smem + kQBytes;
    uint8_t *v_s0 = smem + kQBytes + 2 * kKVBytes;
    uint8_t *p_s = smem + kQBytes + 4 * kKVBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(p_s + BM * BN * 2);
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;   // [2]
    uint64_t *kv_empty = bars + 3;  // [2]
    uint64_t *s_full = bars + 5;    // [2]
    uint64_t *p_full = bars + 7;
    uint64_t *o_done = bars + 8;
    uint32_t &tmem_base_s = *reinterpret_cast<uint32_t *>(bars + 9);
    int &abort_flag = *(reinterpret_cast<int *>(bars + 9) + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y;
    if ((int)blockIdx.x >= __ldg(p.num_entries)) return;
    const int2 ent = p.entries[blockIdx.x];
    const int s = ent.x, tile = ent.y;
    const int q0 = __ldg(p.cu_seqlens_q + s);
    const int q_len = __ldg(p.cu_seqlens_q + s + 1) - q0;
    const int ctx = __ldg(p.context_lens + s);
    if (ctx <= 0 || (int64_t)ctx > (int64_t)p.max_blocks * kB || q_len < 2 || q_len > ctx ||
        q_len > p.max_q_len || q0 < 0 || q0 + q_len > p.total_q) {
        if (tid == 0) set_status(p.status, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int POS = 1 << p.pos_shift;
    const int i0 = tile * POS;
    const int nrows = min(POS, q_len - i0);
    if (nrows <= 0) return;
    const int pos_base = ctx - q_len + i0;
    const int pos_last = pos_base + nrows - 1;
    const int nkv = pos_last / BN + 1;
    const int nb = (ctx + kB - 1) / kB;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) set_status(p.status, PA_ERR_CUDA);
        return;
    }

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(kv_full + i, 1);
            mbar_init(kv_empty + i, 1);
            mbar_init(s_full + i, 1);
        }
        mbar_init(p_full, BM);
        mbar_init(o_done, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&tmem_base_s, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == 4) {
        // ================= TMA producer
        bool ok = true;
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(q_full, kQBytes);
            tma_load_4d(q_s, &tmap_q, 0, q0 + i0, g * p.group, 0, q_full);
        }
        // block ids, 32 per chunk (lane l holds block 32*chunk + l), one chunk ahead;
        // past the sequence end (or invalid) the coordinate num_blocks is out of
        // bounds and TMA fills zeros
        const int32_t *bt = p.block_tables + (int64_t)s * p.max_blocks;
        auto load_ids = [&](int chunk) {
            const int lb = chunk * 32 + lane;
            int coord = p.num_blocks;
            if (lb < nb) {
                const int32_t blk = __ldg(bt + lb);
                if (blk >= 0 && blk < p.num_blocks) coord = blk;
                else set_status(p.status, PA_ERR_OUT_OF_RANGE);
            }
            return coord;
        };
        int ids_cur = load_ids(0), ids_next = load_ids(1), chunk_cur = 0;
        for (int j = 0; j < nkv; ++j) {
            const int stage = j & 1;
            if ((j * kBlocksPerTile) / 32 != chunk_cur) {   // move to the next chunk
                ids_cur = ids_next;
                ++chunk_cur;
                ids_next = load_ids(chunk_cur + 1);
            }
            if (lane == 0 && j >= 2 && !mbar_wait(kv_empty + stage, ((j >> 1) - 1) & 1)) ok = false;
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            int coords[kBlocksPerTile];
            const int lb0 = (j * kBlocksPerTile) & 31;
#pragma unroll
            for (int b = 0; b < kBlocksPerTile; ++b) coords[b] = __shfl_sync(0xffffffffu, ids_cur, lb0 + b);
            // lane 0 arms the barrier, then lanes (block, plane) issue one K and one V copy each
            if (lane == 0) mbar_arrive_expect_tx(kv_full + stage, 2 * kKVBytes);
            __syncwarp();
            if (lane < kBlocksPerTile * kDH) {
                const int b = lane / kDH, dh = lane % kDH;
                int cb = coords[0];
#pragma unroll
                for (int u = 1; u < kBlocksPerTile; ++u) cb = b == u ? coords[u] : cb;
                const uint32_t off = dh * kPlaneKV + b * (kB * 128);
                tma_load_5d(k_s0 + stage * kKVBytes + off, &tmap_k, 0, 0, dh, g, cb, kv_full + stage);
                tma_load_5d(v_s0 + stage * kKVBytes + off, &tmap_v, 0, 0, dh, g, cb, kv_full + stage);
            }
        }
        if (!ok && lane == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            abort_flag = 1;
        }
        // every copy this CTA issued has landed before the CTA may exit
        if (lane == 0) {
            mbar_wait(q_full, 0);
            for (int j = nkv > 2 ? nkv - 2 : 0; j < nkv; ++j) mbar_wait(kv_full + (j & 1), (j >> 1) & 1);
        }
    } else if (warp == 5) {
        // ================= MMA issuer (one thread)
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(q_s), p_addr = smem_u32(p_s);
            auto issue_qk = [&](int j) {
                const uint32_t k_addr = smem_u32(k_s0 + (j & 1) * kKVBytes);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off_q = (ks >> 2) * kPlaneQ + (ks & 3) * 32;
                    const uint32_t off_k = (ks >> 2) * kPlaneKV + (ks & 3) * 32;
                    umma_bf16(tmem + (uint32_t)(j & 1) * kSColStride, umma_desc_sw128(q_addr + off_q, 16, 1024),
                              umma_desc_sw128(k_addr + off_k, 16, 1024), kIdescQK, ks > 0);
                }
            };
            auto issue_pv = [&](int j) {
                const uint32_t v_addr = smem_u32(v_s0 + (j & 1) * kKVBytes);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t off_p = (kk >> 2) * kPlaneQ + (kk & 3) * 32;
                    umma_bf16(tmem + kOCol, umma_desc_sw128(p_addr + off_p, 16, 1024),
                              umma_desc_sw128(v_addr + kk * 2048, kPlaneKV, 1024), kIdescPV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(q_full, 0) && mbar_wait(kv_full, 0);
            if (ok) {
                tc_fence_after();
                issue_qk(0);
                umma_commit(s_full);
            }
            int issued_pv = 0;
            for (int j = 0; ok && j < nkv; ++j) {
                if (j + 1 < nkv) {
                    if (!mbar_wait(kv_full + ((j + 1) & 1), ((j + 1) >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_qk(j + 1);
                    umma_commit(s_full + ((j + 1) & 1));
                }
                if (!mbar_wait(p_full, j & 1)) { ok = false; break; }
                tc_fence_after();
                issue_pv(j);
                umma_commit(o_done);
                umma_commit(kv_empty + (j & 1));
                ++issued_pv;
            }
            if (!ok) {
                set_status(p.status, PA_ERR_TIMEOUT);
                abort_flag = 1;
            }
            // drain: the last product must finish before TMEM is released
            if (issued_pv > 0) mbar_wait(o_done, (issued_pv - 1) & 1);
        }
        __syncwarp();
    } else {
        // ================= softmax warpgroup: thread r owns row r (TMEM lane r)
        const int r = tid;
        const int h_local = r >> p.pos_shift;
        const int i = r & (POS - 1);
        const bool row_valid = i < nrows;
        const int pos = pos_base + (row_valid ? i : nrows - 1);
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        const int t_tail = ctx & (kB - 1);          // valid tokens in the last block (0 = full)
        const int lb_last = (ctx - 1) / kB;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait(s_full + (j & 1), (j >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t raw[BN / 32][32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_addr + (uint32_t)(j & 1) * kSColStride + 32 * c, raw[c]);
            tmem_wait_ld();
            float sv[BN];
            float mx = -INFINITY;
            const int key0 = j * BN;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int key = key0 + 32 * c + e;
                    const float v = key <= pos ? __uint_as_float(raw[c][e]) * p.scale_log2 : -INFINITY;
                    sv[32 * c + e] = v;
                    mx = fmaxf(mx, v);
                }
            const float m_new = fmaxf(m, mx);
            // the running max moves only when it grows by more than 2^8
            const bool need = (j == 0) || m_new > m + 8.f;
            const float m_use_new = need ? m_new : m;
            const float m_use = m_use_new == -INFINITY ? 0.f : m_use_new;
            // P = exp2(S - m) in registers, before waiting for the previous P*V
            float lsum = 0.f;
            uint32_t pw[BN / 2];
#pragma unroll
            for (int u = 0; u < BN / 2; ++u) {
                const float p0 = fast_exp2(sv[2 * u] - m_use);
                const float p1 = fast_exp2(sv[2 * u + 1] - m_use);
                lsum += p0 + p1;
                pw[u] = pack_bf16x2(p0, p1);
            }
            if (j > 0) {
                if (!mbar_wait(o_done, (j - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? fast_exp2(m - m_new) : 1.f;
                    l *= alpha;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(lane_addr + kOCol + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(lane_addr + kOCol + 32 * c, o);
                    }
                    tmem_wait_st();
                }
            }
            m = m_use_new;
            // value rows past the context end inside the last block -> zero
            if (t_tail != 0) {
                const int b = lb_last - j * kBlocksPerTile;
                if (b >= 0 && b < kBlocksPerTile) {
                    if (!mbar_wait(kv_full + (j & 1), (j >> 1) & 1)) { ok = false; break; }
                    uint8_t *vs = v_s0 + (j & 1) * kKVBytes;
                    const int rows_zero = kB - t_tail;
                    const int n16 = kDH * rows_zero * 8;
                    for (int u = r; u < n16; u += BM) {
                        const int dh = u / (rows_zero * 8);
                        const int rem = u - dh * rows_zero * 8;
                        const int tok = t_tail + (rem >> 3);
                        *reinterpret_cast<uint4 *>(vs + dh * kPlaneKV + (b * kB + tok) * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // P as bf16, K-major 128-byte swizzled rows
#pragma unroll
            for (int q4 = 0; q4 < BN / 8; ++q4) {
                const int kt = 8 * q4;                          // first key of this 16-byte chunk
                const int chunk = (kt & 63) >> 3;
                uint8_t *dst = p_s + (kt >> 6) * kPlaneQ + r * 128 + ((chunk ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
            }
            l += lsum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // ---- epilogue: O / l -> bf16 rows of out
        if (ok && mbar_wait(o_done, (nkv - 1) & 1)) {
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16 *dst = p.out + ((int64_t)(q0 + i0 + i) * p.num_heads +
                                          (int64_t)g * p.group + h_local) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_addr + kOCol + 32 * c, o);
                tmem_wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * q4) = v;
                    }
                }
            }
        } else if (!ok) {
            if (r == 0) set_status(p.status, PA_ERR_TIMEOUT);
            abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

CUresult make_q_map(CUtensorMap *map, const void *q, int total_q, int num_heads, int D, int pos,
                    int group) {
    auto encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_FOUND;
    // dims: d_lo(64), row(total_q), head(H), d_hi(D/64); box: 64 x pos x group x D/64
    // -> shared layout [d_hi][head][row][64] = one 128-row K-major operand per plane
    const cuuint64_t dims[4] = {64, (cuuint64_t)total_q, (cuuint64_t)num_heads, (cuuint64_t)(D / 64)};
    const cuuint64_t strides[3] = {(cuuint64_t)num_heads * D * 2, (cuuint64_t)D * 2, 128};
    const cuuint32_t box[4] = {64, (cuuint32_t)pos, (cuuint32_t)group, (cuuint32_t)(D / 64)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult make_kv_map(CUtensorMap *map, const void *pool, int num_blocks, int hkv, int D) {
    auto encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_FOUND;
    // dims: d_lo(64), token(16), d_hi(D/64), head(Hkv), block; box: one block,
    // one head, one 64-column plane -> 16 rows of 128 bytes
    const cuuint64_t dims[5] = {64, (cuuint64_t)kB, (cuuint64_t)(D / 64), (cuuint64_t)hkv,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {(cuuint64_t)hkv * D * 2, 128, (cuuint64_t)D * 2,
                                   (cuuint64_t)kB * hkv * D * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)kB, 1, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int log2_exact(int v) {
    int s = 0;
    while ((1 << s) < v) ++s;
    return (1 << s) == v ? s : -1;
}

template <int D>
cudaError_t launch_main(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                        const PrefillParams &prm, int grid_x, int num_kv_heads, cudaStream_t stream) {
    const size_t smem = (size_t)BM * D * 2 + 4 * (size_t)BN * D * 2 + (size_t)BM * BN * 2 + 128;
    auto kern = prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<dim3(grid_x, num_kv_heads), kThreads, smem, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const AttnArgs &a) {
    if (a.dtype != PA_DTYPE_BF16 || a.block_size != kB) return false;
    if (a.head_dim != 64 && a.head_dim != 128) return false;
    const int G = a.num_heads / a.num_kv_heads;
    if (G > 16 || log2_exact(G) < 0) return false;
    auto al = [](const void *ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
    return al(a.q) && al(a.out) && al(a.k_cache) && al(a.v_cache);
}

size_t prefill_workspace(int num_seqs, int total_q) {
    // plan entries: at most total_q / 8 + num_seqs tiles (8 = fewest positions per tile)
    return align_up(sizeof(int2) * ((size_t)total_q / 8 + num_seqs + 1) + 16, 256);
}

cudaError_t launch_prefill_tc(const AttnArgs &a, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    const int G = a.num_heads / a.num_kv_heads;
    const int pos = BM / G;
    const int pos_shift = log2_exact(pos);
    const int capacity = a.total_q / pos + a.num_seqs;
    if (workspace_bytes < prefill_workspace(a.num_seqs, a.total_q)) return cudaErrorInvalidValue;
    int32_t *count = static_cast<int32_t *>(workspace);
    int2 *entries = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + 16);

    CUtensorMap mq, mk, mv;
    if (make_q_map(&mq, a.q, a.total_q, a.num_heads, a.head_dim, pos, G) != CUDA_SUCCESS ||
        make_kv_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim) != CUDA_SUCCESS ||
        make_kv_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim) != CUDA_SUCCESS)
        return cudaErrorNotSupported;

    prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.cu_seqlens_q, a.num_seqs, pos_shift, entries,
                                                         count, capacity);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    PrefillParams prm;
    prm.cu_seqlens_q = a.cu_seqlens_q;
    prm.context_lens = a.context_lens;
    prm.block_tables = a.block_tables;
    prm.entries = entries;
    prm.num_entries = count;
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.num_seqs = a.num_seqs;
    prm.total_q = a.total_q;
    prm.max_q_len = a.max_q_len;
    prm.num_heads = a.num_heads;
    prm.group = G;
    prm.pos_shift = pos_shift;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    prm.status = a.status;
    return a.head_dim == 64 ? launch_main<64>(mq, mk, mv, prm, capacity, a.num_kv_heads, stream)
                            : launch_main<128>(mq, mk, mv, prm, capacity, a.num_kv_heads, stream);
}

}  // namespace pa
