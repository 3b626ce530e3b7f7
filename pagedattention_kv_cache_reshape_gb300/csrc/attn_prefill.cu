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
// Work unit (one CTA): two M-tiles of 128 rows; a tile is POS consecutive
// query positions x the G query heads of one kv-head, so each K/V tile is
// loaded once for 2*POS positions of the whole group.  Keys come in tiles of
// 64 (4 cache blocks) through a 3-deep TMA ring.
// Warp roles: warps 0-7 two softmax warpgroups (thread = row = TMEM lane of
// its tile), warp 8 TMA producer, warp 9 TMEM owner and MMA issuer.
//   S_t,j = Q_t K_j^T  -> TMEM (two buffers per tile)
//   P_t,j = exp2(S_t,j * scale*log2e - m)  (bf16, shared memory, two buffers)
//   O_t  += P_t,j V_j  -> TMEM (fp32)
// The issuer runs QK of KV tile j for both M-tiles before PV of tile j-1, so
// the tensor pipe has work while the softmax warpgroups turn S into P.
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
constexpr int BM = 128;               // rows per M-tile
constexpr int kMT = 2;                // M-tiles per CTA, one softmax warpgroup each
constexpr int BN = 64;                // keys per KV tile (4 cache blocks)
constexpr int kStages = 3;            // K/V ring depth
constexpr int kBlocksPerTile = BN / kB;
constexpr int kProducerWarp = 4 * kMT;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kPlanThreads = 512;
constexpr int kTmemCols = 512;

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
    int causal;      // 0: encode-only, every row sees the whole sequence
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
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    constexpr int kDH = D / 64;             // 64-column planes of a head
    constexpr int kQBytes = BM * D * 2;     // one M-tile of Q
    constexpr int kKVBytes = BN * D * 2;    // K (or V) of one KV tile
    constexpr int kPBytes = BM * BN * 2;    // one P buffer
    constexpr int kPlaneQ = BM * 128;       // one 64-column plane of Q or P
    constexpr int kPlaneKV = BN * 128;      // one 64-column plane of K or V
    constexpr uint32_t kIdescQK = umma_idesc_bf16(BM, BN, 0);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(BM, D, 1);

    // all shared state is dynamic so the 1024-byte aligned tiles start at 0:
    // Q[2] | (K,V) x kStages | P[2 tiles][2 buffers] | barriers
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *q_s = smem;
    uint8_t *kv_s = smem + kMT * kQBytes;
    uint8_t *p_s = kv_s + kStages * 2 * kKVBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(p_s + kMT * 2 * kPBytes);
    uint64_t *q_full = bars;                       // 1
    uint64_t *kv_full = q_full + 1;                // [kStages]
    uint64_t *kv_empty = kv_full + kStages;        // [kStages]
    uint64_t *s_full = kv_empty + kStages;         // [tile][buf]
    uint64_t *p_full = s_full + 4;                 // [tile][buf]
    uint64_t *p_free = p_full + 4;                 // [tile][buf]
    uint64_t *drained = p_free + 4;                // 1: every product issued has completed
    uint32_t &tmem_base_s = *reinterpret_cast<uint32_t *>(drained + 1);
    int &abort_flag = *(reinterpret_cast<int *>(drained + 1) + 1);

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
    const int POS = 1 << p.pos_shift;                  // query positions per M-tile
    const int i0 = tile * kMT * POS;                   // first position of M-tile 0
    const int nrows_all = min(kMT * POS, q_len - i0);  // valid positions of the CTA
    if (nrows_all <= 0) return;
    const int pos_base = ctx - q_len + i0;
    const int pos_last = p.causal ? pos_base + nrows_all - 1 : ctx - 1;
    const int nkv = pos_last / BN + 1;
    const int nb = (ctx + kB - 1) / kB;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) set_status(p.status, PA_ERR_CUDA);
        return;
    }

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(kv_full + i, 1);
            mbar_init(kv_empty + i, 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(p_full + i, BM);
            mbar_init(p_free + i, 1);
        }
        mbar_init(drained, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(&tmem_base_s, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    // TMEM columns: S[tile][buf] at (2 tile + buf) * BN, O[tile] at 4 BN + tile * D
    auto s_col = [](int t, int b) { return (uint32_t)((2 * t + b) * BN); };
    auto o_col = [](int t) { return (uint32_t)(4 * BN + t * D); };

    if (warp == kProducerWarp) {
        // ================= TMA producer
        bool ok = true;
        if (lane == 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(q_full, kMT * kQBytes);
            for (int t = 0; t < kMT; ++t)
                tma_load_4d(q_s + t * kQBytes, &tmap_q, 0, q0 + i0 + t * POS, g * p.group, 0, q_full);
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
            const int stage = j % kStages;
            if ((j * kBlocksPerTile) / 32 != chunk_cur) {
                ids_cur = ids_next;
                ++chunk_cur;
                ids_next = load_ids(chunk_cur + 1);
            }
            if (lane == 0 && j >= kStages && !mbar_wait(kv_empty + stage, ((j / kStages) - 1) & 1)) ok = false;
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
                uint8_t *ks = kv_s + stage * 2 * kKVBytes;
                tma_load_5d(ks + off, &tmap_k, 0, 0, dh, g, cb, kv_full + stage);
                tma_load_5d(ks + kKVBytes + off, &tmap_v, 0, 0, dh, g, cb, kv_full + stage);
            }
        }
        if (!ok && lane == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            abort_flag = 1;
        }
        // every copy this CTA issued has landed before the CTA may exit
        if (lane == 0) {
            mbar_wait(q_full, 0);
            for (int j = nkv > kStages ? nkv - kStages : 0; j < nkv; ++j)
                mbar_wait(kv_full + (j % kStages), (j / kStages) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer (one thread): QK of KV tile j for both
        // M-tiles, then PV of tile j-1, so the tensor pipe has work while the
        // softmax warpgroups turn S into P
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(q_s), p_addr = smem_u32(p_s), kv_addr = smem_u32(kv_s);
            auto issue_qk = [&](int t, int j) {
                const uint32_t k_addr = kv_addr + (j % kStages) * 2 * kKVBytes;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off_q = t * kQBytes + (ks >> 2) * kPlaneQ + (ks & 3) * 32;
                    const uint32_t off_k = (ks >> 2) * kPlaneKV + (ks & 3) * 32;
                    umma_bf16(tmem + s_col(t, j & 1), umma_desc_sw128(q_addr + off_q, 16, 1024),
                              umma_desc_sw128(k_addr + off_k, 16, 1024), kIdescQK, ks > 0);
                }
            };
            auto issue_pv = [&](int t, int j) {
                const uint32_t v_addr = kv_addr + (j % kStages) * 2 * kKVBytes + kKVBytes;
                const uint32_t pb = p_addr + (2 * t + (j & 1)) * kPBytes;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t off_p = (kk >> 2) * kPlaneQ + (kk & 3) * 32;
                    umma_bf16(tmem + o_col(t), umma_desc_sw128(pb + off_p, 16, 1024),
                              umma_desc_sw128(v_addr + kk * 2048, kPlaneKV, 1024), kIdescPV,
                              (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto pv_step = [&](int j) -> bool {   // PV of KV tile j for both M-tiles
                for (int t = 0; t < kMT; ++t) {
                    if (!mbar_wait(p_full + 2 * t + (j & 1), (j >> 1) & 1)) return false;
                    tc_fence_after();
                    issue_pv(t, j);
                    umma_commit(p_free + 2 * t + (j & 1));
                }
                umma_commit(kv_empty + (j % kStages));
                return true;
            };
            bool ok = mbar_wait(q_full, 0);
            int pv_issued = 0;
            for (int j = 0; ok && j < nkv; ++j) {
                if (!mbar_wait(kv_full + (j % kStages), (j / kStages) & 1)) { ok = false; break; }
                tc_fence_after();
                for (int t = 0; t < kMT; ++t) {
                    issue_qk(t, j);
                    umma_commit(s_full + 2 * t + (j & 1));
                }
                if (j >= 1) {
                    if (!pv_step(j - 1)) { ok = false; break; }
                    ++pv_issued;
                }
            }
            if (ok) {
                if (pv_step(nkv - 1)) ++pv_issued;
                else ok = false;
            }
            if (!ok) {
                set_status(p.status, PA_ERR_TIMEOUT);
                abort_flag = 1;
            }
            // drain: everything issued must finish before TMEM is released
            umma_commit(drained);
            mbar_wait(drained, 0);
            (void)pv_issued;
        }
        __syncwarp();
    } else {
        // ================= softmax warpgroup t: thread r owns row r of M-tile t
        const int t = warp >> 2;
        const int r = tid & (BM - 1);
        const int h_local = r >> p.pos_shift;
        const int i = t * POS + (r & (POS - 1));          // position index within the CTA
        const bool row_valid = i < nrows_all;
        // last visible key of this row: its position (causal) or the sequence end
        const int pos = p.causal ? pos_base + (row_valid ? i : nrows_all - 1) : ctx - 1;
        const int first_pos = p.causal ? pos_base + t * POS : ctx - 1;   // smallest pos of the tile
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int t_tail = ctx & (kB - 1);          // valid tokens in the last block (0 = full)
        const int lb_last = (ctx - 1) / kB;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            const int b = j & 1;
            if (!mbar_wait(s_full + 2 * t + b, (j >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t raw[BN / 32][32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_addr + s_col(t, b) + 32 * c, raw[c]);
            tmem_wait_ld();
            float sv[BN];
            float mx = -INFINITY;
            const int key0 = j * BN;
            const bool diag = key0 + BN - 1 > first_pos;   // a key past some row of this tile
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = __uint_as_float(raw[c][e]) * p.scale_log2;
                    const float v = (!diag || key0 + 32 * c + e <= pos) ? x : -INFINITY;
                    sv[32 * c + e] = v;
                    mx = fmaxf(mx, v);
                }
            const float m_new = fmaxf(m, mx);
            // the running max moves only when it grows by more than 2^8
            const bool need = (j == 0) || m_new > m + 8.f;
            const float m_use_new = need ? m_new : m;
            const float m_use = m_use_new == -INFINITY ? 0.f : m_use_new;
            float lsum = 0.f;
            uint32_t pw[BN / 2];
#pragma unroll
            for (int u = 0; u < BN / 2; ++u) {
                const float p0 = fast_exp2(sv[2 * u] - m_use);
                const float p1 = fast_exp2(sv[2 * u + 1] - m_use);
                lsum += p0 + p1;
                pw[u] = pack_bf16x2(p0, p1);
            }
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O must hold every earlier product before it is rescaled: wait
                // for the commit of PV(j-1) on its P buffer (that barrier is at
                // most one phase ahead of this wait, so its parity is exact;
                // a commit also covers every earlier product)
                if (!mbar_wait(p_free + 2 * t + ((j - 1) & 1), ((j - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const float alpha = need ? fast_exp2(m - m_new) : 1.f;
                l *= alpha;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + o_col(t) + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(lane_addr + o_col(t) + 32 * c, o);
                }
                tmem_wait_st();
            }
            m = m_use_new;
            // value rows past the context end inside the last block -> zero
            // (warpgroup 0 only; its p_full arrival orders the writes before
            // every product of this KV tile)
            if (t == 0 && t_tail != 0) {
                const int bb = lb_last - j * kBlocksPerTile;
                if (bb >= 0 && bb < kBlocksPerTile) {
                    if (!mbar_wait(kv_full + (j % kStages), (j / kStages) & 1)) { ok = false; break; }
                    uint8_t *vs = kv_s + (j % kStages) * 2 * kKVBytes + kKVBytes;
                    const int rows_zero = kB - t_tail;
                    const int n16 = kDH * rows_zero * 8;
                    for (int u = r; u < n16; u += BM) {
                        const int dh = u / (rows_zero * 8);
                        const int rem = u - dh * rows_zero * 8;
                        const int tok = t_tail + (rem >> 3);
                        *reinterpret_cast<uint4 *>(vs + dh * kPlaneKV + (bb * kB + tok) * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // the P buffer is free once the product two tiles back has read it
            if (j >= 2 && !mbar_wait(p_free + 2 * t + b, ((j >> 1) - 1) & 1)) { ok = false; break; }
            uint8_t *pbuf = p_s + (2 * t + b) * kPBytes;
#pragma unroll
            for (int q4 = 0; q4 < BN / 8; ++q4) {
                const int kt = 8 * q4;                          // first key of this 16-byte chunk
                const int chunk = (kt & 63) >> 3;
                uint8_t *dst = pbuf + (kt >> 6) * kPlaneQ + r * 128 + ((chunk ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
            }
            l += lsum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full + 2 * t + b);
        }
        // ---- epilogue: O / l -> bf16 rows of out, after the commit of the last product
        if (ok && mbar_wait(p_free + 2 * t + ((nkv - 1) & 1), ((nkv - 1) >> 1) & 1)) {
            tc_fence_after();
            const float inv = 1.f / l;
            __nv_bfloat16 *dst = p.out + ((int64_t)(q0 + i0 + i) * p.num_heads +
                                          (int64_t)g * p.group + h_local) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_addr + o_col(t) + 32 * c, o);
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
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
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
    const size_t smem = (size_t)kMT * BM * D * 2 + (size_t)kStages * 2 * BN * D * 2 +
                        (size_t)kMT * 2 * BM * BN * 2 + 256;
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
    const int cta_shift = pos_shift + 1;          // kMT = 2 M-tiles of `pos` positions per CTA
    const int capacity = a.total_q / (kMT * pos) + a.num_seqs;
    if (workspace_bytes < prefill_workspace(a.num_seqs, a.total_q)) return cudaErrorInvalidValue;
    int32_t *count = static_cast<int32_t *>(workspace);
    int2 *entries = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + 16);

    CUtensorMap mq, mk, mv;
    if (make_q_map(&mq, a.q, a.total_q, a.num_heads, a.head_dim, pos, G) != CUDA_SUCCESS ||
        make_kv_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim) != CUDA_SUCCESS ||
        make_kv_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim) != CUDA_SUCCESS)
        return cudaErrorNotSupported;

    prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.cu_seqlens_q, a.num_seqs, cta_shift, entries,
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
    prm.causal = a.causal;
    return a.head_dim == 64 ? launch_main<64>(mq, mk, mv, prm, capacity, a.num_kv_heads, stream)
                            : launch_main<128>(mq, mk, mv, prm, capacity, a.num_kv_heads, stream);
}

}  // namespace pa
