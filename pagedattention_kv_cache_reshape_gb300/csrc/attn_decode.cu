// attn_decode.cu -- persistent split-KV paged decode for bf16 caches.
//
// What it computes ("vLLM：颠覆大模型推理的高效API服务引擎深度解析" §1.3:
// attention gathers the scattered physical blocks through the block table;
// "vLLM изнутри…", model-runner paragraph: decode reads earlier tokens' KV
// from the cache and is memory-bound): for every sequence s and q-head h,
//     out[s][h] = sum_j softmax_j(scale * <q[s][h], K_s[j][g(h)]>) V_s[j][g(h)].
//
// How (the design is this library's own, built around HBM streaming):
//  * plan kernel -- from context_lens, an exclusive prefix over the number of
//    16-token blocks each sequence needs, and one 16-byte entry per logical
//    block of the whole batch (sequence, query row, physical block id, valid
//    tokens).  The batch becomes one stream of T blocks; with NHG kv-head
//    groups the virtual stream has NHG*T entries.
//  * main kernel -- one persistent CTA per SM takes an equal contiguous slice
//    of the virtual stream, so every CTA reads the same number of cache bytes
//    whatever the length mix.  A producer warp loads each 16-token unit of
//    KVH kv-heads (32 KB of K and 32 KB of V for 8 heads x 128 dims) with one
//    TMA tensor copy each (two at block size 8) into a ring of shared-memory
//    stages (128-byte swizzle), plus the sequence's query heads when a new
//    sequence starts.
//    A consumer warp owns up to 8 q-heads of one kv-head (a kv-head with G > 8
//    q-heads gets ceil(G/8) warps): S^T = K Q^T and O^T += V^T P^T run on the
//    tensor cores (mma m16n8k16, bf16 in, fp32 out), the unit's 16 tokens in
//    M and the q-heads in N, with an online softmax (running max / sum,
//    base-2 exponent) in fp32.
//    A sequence slice wholly inside one CTA is normalised and stored.  A
//    sequence cut by CTA boundaries leaves (m, l, o) partials; the warp that
//    stores the last of a sequence's pieces (an arrival counter per cut and
//    kv-head, zeroed by the plan) merges them in CTA order:
//        M = max m_i, L = sum l_i 2^{m_i - M}, o = sum 2^{m_i - M} o_i / L.
// The two kernels are launched as programmatic dependents: the main kernel is
// resident early and waits (griddepcontrol.wait) for the plan only after its
// prologue, so launch latency overlaps the plan.
// Every cache byte is read once from HBM; the partition depends only on
// context_lens and the CTA count, and the merge order is fixed, so results
// are bitwise reproducible and do not depend on which physical blocks hold
// the data or which CTA finishes first.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <utility>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// The decode streams 16-token units whatever the cache block size B (8, 16
// or 32 tokens): a unit is one block at B = 16, half a block at B = 32 (one
// TMA box at token offset 0 or 16) and two blocks at B = 8 (two 8-row boxes;
// the consumer's ldmatrix rows address both).  A unit is a stage of the ring
// and the M of the consumer's m16n8k16 products.
constexpr int kU = 16;
constexpr int kMaxKvhPerCta = 8;
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxQHeadsPerCta = 32;
constexpr int kHeadsPerWarp = 8;    // the N of one m16n8k16 product: q-heads per consumer warp
constexpr int kMaxGroup = 32;       // q-heads per kv-head
constexpr int kMaxSeqs = 16384;     // prefix of all sequences kept in shared memory
constexpr int kMaxSeqsEarlyPrefetch = 4096;   // the early prefetch reads every context length: bounded
constexpr int kPartialCtas = 512;   // partial slots reserved for CTA boundaries
constexpr int kPlanThreads = 256;
constexpr int kSmemBudget = 227 * 1024;
// Per-SM rates for splitting the SMs between the decode rows and a concurrent
// prefill kernel (GB300): the tcgen05 prefill kernel sustains about 7.6
// TFLOP/s per SM on causal chunks alone, but beside the decode kernel the
// split balances best at 6.6 (a sweep of 5.9-8.2 on the 8 x 512 + 248-row mixed
// batch); the decode kernel streams up to about 82 GB/s from one SM alone,
// and the split balances best at 64 GB/s per SM: a sweep of 50-88 put the step
// at its shortest between 58 and 70.
constexpr double kDecodeBytesPerSmNs = 64.0;
constexpr double kPrefillFlopsPerSmNs = 6600.0;

struct __align__(16) StreamEntry {
    int32_t seq;
    int32_t qrow;    // query / output row of the sequence
    int32_t blk;     // physical block id (B = 8: the unit's first block), -1 if a table entry was invalid
    int32_t packed;  // ntok (bits 0..5) | last unit of its sequence (bit 6) | B = 32: upper half (bit 7) | unit << 8
};

struct __align__(16) StageHeader {
    int32_t seq, qrow, hg, lb, ntok, flags, pad0, pad1;
};
constexpr int kFirst = 1, kLast = 2, kSeqEnd = 4, kValid = 8;

struct DecodeParams {
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    const int32_t *prefix;     // [num_seqs + 1]
    const StreamEntry *stream; // [T]
    const int32_t *stream_b1;  // [T], B = 8 only: the unit's second block (-1: past the sequence end)
    int log2b;                 // log2 of the cache block size
    float *part_o;             // [slots][QH][D]
    float *part_ml;            // [slots][QH][2]
    int num_seqs;
    int num_heads;
    int kvh;       // kv-heads per CTA
    int wpk;       // consumer warps per kv-head: ceil(group / 8)
    int gw;        // q-heads per consumer warp: ceil(group / wpk)
    int group;     // q-heads per kv-head
    int qh;        // q-heads per CTA = kvh * group
    int nhg;       // kv-head groups
    int32_t *arrivals;         // [CTAs][consumer warps] arrival counters of cut sequences, zeroed by the plan
    const int32_t *active;     // CTAs that take a slice (written by the plan; the rest exit)
    int shared_sms;            // 1: `active` is set (a prefill kernel shares the SMs); 0: all CTAs
    int num_stages;
    int tma_heads; // kv-heads per TMA op (kvh, or 1 with the per-head map)
    float scale_log2;
    int32_t *status;
    // for the L2 prefetch of the CTA's first blocks while it waits for the
    // plan (decode calls without cu_seqlens_q only; null context_lens: none)
    const int32_t *context_lens;
    const int32_t *block_tables;
    int max_blocks;
    int num_blocks;
    int num_kv_heads;
    const uint8_t *k_bytes, *v_bytes;   // the pools
    // bounded waits: their limit, and the test hook's stall (PA_STALL_*)
    uint64_t wait_ns;
    int stall;
    int stall_after;
    int32_t *wait_sites;
};

// Optional cache write folded into the plan kernel (pa_decode_step): for new
// token t of sequence s (cu_new[s] <= t < cu_new[s+1]) at position
// p = seq_start[s] + t - cu_new[s], slot = block_tables[s][p/B]*B + p%B;
// the token's K and V rows are copied there with 16-byte vectors.
struct KvWriteJob {
    const int32_t *seq_start;
    const int32_t *cu_new;
    int total_new;
    const uint4 *key;
    const uint4 *value;
    int64_t key_stride_v;    // token strides in 16-byte vectors
    int64_t value_stride_v;
    uint4 *k_cache;
    uint4 *v_cache;
    int64_t *slot_mapping;
    int row_vecs;            // 16-byte vectors per token row
    int64_t pool_slots;
    int first_cta;           // the plan launch's CTAs from here on do the write
};

// How many of the decode kernel's CTAs take a slice.  Alone on the GPU,
// every CTA does.  Beside the tensor-core prefill of the same batch (which
// runs concurrently and takes over the SMs the decode kernel leaves), the
// SMs are split by estimated work: decode blocks at the per-SM streaming
// rate against the causal (query, key) pairs of the prefill rows at the
// per-SM tensor rate, both measured on GB300.
struct DecodeSplit {
    int32_t *active;
    int32_t *arrivals;  // zeroed by the plan: [num_arrivals]
    int num_arrivals;
    int grid;          // CTAs the decode kernel is launched with
    int share;         // 1: a prefill kernel runs beside this one
    int causal;
    double block_ns;   // SM-nanoseconds per decode block of all kv-heads
    double pair_ns;    // SM-nanoseconds per causal (query row, key) pair of all heads
};

// ------------------------------------------------------------------ plan
// CTAs [0, job.first_cta) build the block stream (CTA 0 also zeroes the
// arrival counters); the CTAs after them, up to the last, write the step's
// new tokens into the cache, concurrently.  kShare: the batch also has
// prefill chunks (the last CTA plans them and CTA 0 sets the SM split);
// decode-only calls run the plain instantiation.
template <bool kShare>
__global__ void __launch_bounds__(kPlanThreads)
    decode_plan_kernel(const int32_t *__restrict__ context_lens,
                       const int32_t *__restrict__ cu_seqlens_q,
                       const int32_t *__restrict__ block_tables, int num_seqs, int max_blocks,
                       int num_blocks, int total_q, int log2b, int32_t *__restrict__ prefix,
                       StreamEntry *__restrict__ stream, int32_t *__restrict__ stream_b1, int32_t *status,
                       const KvWriteJob job,
                       const DecodeSplit split, const PrefillPlanJob prefill) {
    const int B = 1 << log2b;   // tokens per cache block
    extern __shared__ __align__(16) int32_t pref_s[];  // [num_seqs + 1]
    __shared__ int32_t warp_tot[kPlanThreads / 32];
    __shared__ double pair_tot[kPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependency_wait();      // inputs may come from the previous kernel
    grid_dependents_launch();    // the decode kernel may start its prologue
    // with prefill chunks in the batch, the last CTA builds their work list
    const int dgrid = (int)gridDim.x - (kShare ? 1 : 0);   // CTAs of the plan and the cache write
    if (kShare && (int)blockIdx.x == dgrid) {
        prefill_plan_block(prefill, reinterpret_cast<uint8_t *>(pref_s));
        return;
    }
    if (blockIdx.x == 0)
        for (int i = tid; i < split.num_arrivals; i += kPlanThreads) split.arrivals[i] = 0;
    if ((int)blockIdx.x >= job.first_cta) {
        // ---- the step's cache write, beside the plan.  Work item = one chunk of
        // up to 32 * kPre 16-byte vectors of one new token's K and V rows, so a
        // wide row (32 kv-heads x 128 dims = 512 vectors) is spread over several
        // warps and every warp's loads are in flight together before its stores.
        const int warps = kPlanThreads / 32;
        const int wctas = dgrid - job.first_cta;
        constexpr int kPre = 4;   // vectors per lane per item
        constexpr int kChunk = 32 * kPre;
        const int chunks = (job.row_vecs + kChunk - 1) / kChunk;
        const int64_t items = (int64_t)job.total_new * chunks;
        for (int64_t it = (int64_t)((int)blockIdx.x - job.first_cta) * warps + warp; it < items;
             it += (int64_t)wctas * warps) {
            const int t = (int)(it / chunks);
            const int v0 = (int)(it - (int64_t)t * chunks) * kChunk;
            const uint4 *ks = job.key + t * job.key_stride_v;
            const uint4 *vs = job.value + t * job.value_stride_v;
            // the rows depend only on t: their loads overlap the slot's dependent loads
            uint4 kr[kPre], vr[kPre];
#pragma unroll
            for (int u = 0; u < kPre; ++u) {
                const int i = v0 + lane + 32 * u;
                if (i < job.row_vecs) {
                    kr[u] = __ldg(ks + i);
                    vr[u] = __ldg(vs + i);
                }
            }
            int64_t slot = -1;
            if (lane == 0) {
                // the token's sequence: s = t when sequence t has exactly its one new
                // token at t (checked), else the last s with cu_new[s] <= t
                int s = -1, c0 = 0, st = 0;
                if (t < num_seqs) {
                    c0 = __ldg(job.cu_new + t);
                    const int c1 = __ldg(job.cu_new + t + 1);
                    st = __ldg(job.seq_start + t);
                    if (c0 <= t && t < c1) s = t;
                }
                if (s < 0) {
                    int lo = 0, hi = num_seqs;
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (__ldg(job.cu_new + mid) <= t) lo = mid; else hi = mid;
                    }
                    s = lo;
                    c0 = __ldg(job.cu_new + lo);
                    st = __ldg(job.seq_start + lo);
                }
                const int64_t pos = (int64_t)st + (t - c0);
                const int64_t logical = pos >> log2b;
                // every chunk of the token finds the same slot; the first records it
                if (pos < 0 || logical >= max_blocks) {
                    if (v0 == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
                } else {
                    const int32_t phys = __ldg(block_tables + (int64_t)s * max_blocks + logical);
                    if (phys < 0 || phys >= num_blocks) {
                        if (v0 == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
                    } else {
                        slot = ((int64_t)phys << log2b) + (pos - (logical << log2b));
                    }
                }
                if (v0 == 0) job.slot_mapping[t] = slot;
            }
            slot = __shfl_sync(0xffffffffu, slot, 0);
            if (slot < 0 || slot >= job.pool_slots) continue;
            uint4 *kd = job.k_cache + slot * job.row_vecs;
            uint4 *vd = job.v_cache + slot * job.row_vecs;
#pragma unroll
            for (int u = 0; u < kPre; ++u) {
                const int i = v0 + lane + 32 * u;
                if (i < job.row_vecs) {
                    kd[i] = kr[u];
                    vd[i] = vr[u];
                }
            }
        }
        return;
    }
    const int pgrid = job.first_cta;   // CTAs of the plan proper
    int running = 0;
    double pairs = 0.0;   // causal (query, key) pairs of this thread's prefill rows
    for (int base = 0; base < num_seqs; base += kPlanThreads) {
        const int s = base + tid;
        int nb = 0;
        if (s < num_seqs) {
            const int q0 = cu_seqlens_q ? __ldg(cu_seqlens_q + s) : s;
            const int q1 = cu_seqlens_q ? __ldg(cu_seqlens_q + s + 1) : s + 1;
            const int q_len = q1 - q0;
            const int ctx = __ldg(context_lens + s);
            if (kShare && q_len >= 2 && q_len <= ctx)
                pairs += split.causal ? (double)q_len * (ctx - q_len) + 0.5 * (double)q_len * (q_len + 1)
                                      : (double)q_len * ctx;
            if (q0 < 0 || q1 < q0 || q1 > total_q) {
                if (blockIdx.x == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
            } else if (q_len == 1) {
                if (ctx <= 0 || (int64_t)ctx > (int64_t)max_blocks * B) {
                    if (blockIdx.x == 0) set_status(status, PA_ERR_OUT_OF_RANGE);
                } else {
                    nb = (ctx + kU - 1) / kU;   // 16-token units
                }
            }
        }
        int incl = nb;  // inclusive warp scan
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int warp_off = 0, chunk_tot = 0;
        for (int w = 0; w < kPlanThreads / 32; ++w) {
            const int t = warp_tot[w];
            if (w < warp) warp_off += t;
            chunk_tot += t;
        }
        if (s < num_seqs) pref_s[s] = running + warp_off + incl - nb;
        running += chunk_tot;
        __syncthreads();
    }
    if (tid == 0) pref_s[num_seqs] = running;
    if (kShare && blockIdx.x == 0) {
        // CTAs of the decode kernel that take a slice
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) pairs += __shfl_xor_sync(0xffffffffu, pairs, off);
        if (lane == 0) pair_tot[warp] = pairs;
        __syncthreads();
        if (tid == 0) {
            int act = split.grid;
            {
                double pf = 0.0;
                for (int w = 0; w < kPlanThreads / 32; ++w) pf += pair_tot[w];
                const double dec = (double)running * split.block_ns;
                pf *= split.pair_ns;
                if (pf > 0.0 && dec > 0.0) {
                    act = (int)llrint(split.grid * dec / (dec + pf));
                    act = act < 1 ? 1 : (act > split.grid ? split.grid : act);
                }
            }
            *split.active = act;
        }
    }
    __syncthreads();
    const int T = running;
    if (blockIdx.x == 0)
        for (int s = tid; s <= num_seqs; s += kPlanThreads) prefix[s] = pref_s[s];
    for (int b = blockIdx.x * kPlanThreads + tid; b < T; b += pgrid * kPlanThreads) {
        int lo = 0, hi = num_seqs;  // last s with pref_s[s] <= b
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pref_s[mid] <= b) lo = mid; else hi = mid;
        }
        const int s = lo;
        const int lb = b - pref_s[s];            // 16-token unit of the sequence
        const int ctx = __ldg(context_lens + s);
        const int32_t *row = block_tables + (int64_t)s * max_blocks;
        // the unit's physical block(s): B = 16 one, B = 32 half of one, B = 8 two
        // (the second -1 past the sequence end; an invalid entry voids the unit)
        int32_t blk, blk1 = -1;
        int half = 0;
        if (log2b == 4) {
            blk = __ldg(row + lb);
        } else if (log2b == 5) {
            blk = __ldg(row + (lb >> 1));
            half = lb & 1;
        } else {
            blk = __ldg(row + 2 * lb);
            if ((2 * lb + 1) * 8 < ctx) {
                blk1 = __ldg(row + 2 * lb + 1);
                if (blk1 < 0 || blk1 >= num_blocks) blk = num_blocks;   // voids the unit below
            }
        }
        if (blk < 0 || blk >= num_blocks) {
            set_status(status, PA_ERR_OUT_OF_RANGE);
            blk = -1;
        }
        const int ntok = min(kU, ctx - lb * kU);
        const int seq_end = (lb + 1) * kU >= ctx ? 1 : 0;
        StreamEntry e;
        e.seq = s;
        e.qrow = cu_seqlens_q ? __ldg(cu_seqlens_q + s) : s;
        e.blk = blk;
        e.packed = ntok | (seq_end << 6) | (half << 7) | (lb << 8);
        stream[b] = e;
        if (log2b == 3) stream_b1[b] = blk1;
    }
}

__device__ __forceinline__ int64_t cta_slice_begin(int64_t c, int64_t nv, int64_t p) {
    return c * nv / p;
}
// CTA whose slice holds virtual block v.
__device__ __forceinline__ int64_t cta_of(int64_t v, int64_t nv, int64_t p) {
    return ((v + 1) * p - 1) / nv;
}

// ------------------------------------------------------------------ merge
// One warp merges the pieces of a cut sequence for nh <= 4 q-heads h0.. of
// its kv-head group (lane: D/32 consecutive dims of each), in CTA order
// c0..c1, with the online rule (M, L, acc) <- (max, L a + l b, acc a + o b),
// a = 2^{M - M'}, b = 2^{m - M'}, per head.  The loads of two pieces of all
// nh heads are in flight at a time.  The partials were written by other
// SMs: they are read through L2.
template <int D>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, int64_t vs, int64_t c0,
                                             int64_t c1, int64_t NV, int64_t P, int h0, int nh,
                                             __nv_bfloat16 *dst) {
    constexpr int kPer = D / 32;
    constexpr int kH = 4;
    constexpr int kBatch = 2;
    const int lane = threadIdx.x & 31;
    float M[kH], L[kH], acc[kH][kPer];
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
        M[hh] = -INFINITY;
        L[hh] = 0.f;
#pragma unroll
        for (int u = 0; u < kPer; ++u) acc[hh][u] = 0.f;
    }
    for (int64_t cb = c0; cb <= c1; cb += kBatch) {
        float2 ml[kBatch][kH];
        float ov[kBatch][kH][kPer];
        bool use[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int64_t c = cb + k;
            // CTAs with an empty slice (fewer blocks than CTAs) hold no piece
            use[k] = c <= c1 && (NV >= P || cta_slice_begin(c, NV, P) < cta_slice_begin(c + 1, NV, P));
            const int64_t slot = vs + (use[k] ? c : c0);
#pragma unroll
            for (int hh = 0; hh < kH; ++hh) {
                const int h_loc = h0 + (hh < nh ? hh : 0);
                ml[k][hh] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (slot * p.qh + h_loc) * 2));
                const float *src = p.part_o + (slot * p.qh + h_loc) * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    ov[k][hh][0] = t.x; ov[k][hh][1] = t.y; ov[k][hh][2] = t.z; ov[k][hh][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    ov[k][hh][0] = t.x; ov[k][hh][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
            for (int hh = 0; hh < kH; ++hh) {
                if (!use[k] || ml[k][hh].x == -INFINITY) continue;
                const float Mn = fmaxf(M[hh], ml[k][hh].x);
                const float a = fast_exp2(M[hh] - Mn), b = fast_exp2(ml[k][hh].x - Mn);
                L[hh] = L[hh] * a + ml[k][hh].y * b;
#pragma unroll
                for (int u = 0; u < kPer; ++u) acc[hh][u] = acc[hh][u] * a + ov[k][hh][u] * b;
                M[hh] = Mn;
            }
    }
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
        if (hh >= nh) break;
        const float inv = 1.f / L[hh];
#pragma unroll
        for (int u = 0; u < kPer; u += 2)
            *reinterpret_cast<uint32_t *>(dst + hh * D + lane * kPer + u) =
                pack_bf16x2(acc[hh][u] * inv, acc[hh][u + 1] * inv);
    }
}

// ------------------------------------------------------------------ tree merge
// A sequence cut into many pieces (a few long sequences spread over all
// CTAs) is merged up a fixed 4-ary tree over its pieces' local indices
// i = c - c0 (0..n-1), as the pieces arrive: at level l the group g holds the
// children g 4^{l+1} + m 4^l (m = 0..3, those < n) and one counter; the warp
// that brings the counter to the group's child count merges the children in
// order into the first child's slot (merge_pieces' online rule) and goes on
// up, so about log4(n) merges follow the last piece instead of n.  The tree
// is fixed, so results do not depend on which piece arrives first.
// Counters: the unit's group j (groups with two or more children, counted
// level by level) at c0 + j < c1, so units never share one.
constexpr int kTreeMinPieces = 16;
constexpr int kTreeFan = 4;

// groups with two or more children at level m of the tree over n leaves
__device__ __forceinline__ int tree_groups(int m, int n) {
    const int child = 1 << (2 * m), span = child << 2;   // 4^m, 4^{m+1}
    return n > child ? (n - child + span - 1) / span : 0;
}

// Children base, base + stride, ... (cnt of them, slots vs + c0 + index) merged
// in order for nh <= 4 q-heads h0..; into the first child's slot, or, with
// `dst`, normalised into the output rows.
template <int D>
__device__ __forceinline__ void merge_group(const DecodeParams &p, int64_t slot0, int stride, int cnt, int h0,
                                            int nh, __nv_bfloat16 *dst) {
    constexpr int kPer = D / 32;
    constexpr int kH = 4;
    const int lane = threadIdx.x & 31;
    float M[kH], L[kH], acc[kH][kPer];
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
        M[hh] = -INFINITY;
        L[hh] = 0.f;
#pragma unroll
        for (int u = 0; u < kPer; ++u) acc[hh][u] = 0.f;
    }
    for (int k0 = 0; k0 < cnt; k0 += 2) {
        float2 ml[2][kH];
        float ov[2][kH][kPer];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int64_t slot = slot0 + (int64_t)(k0 + k < cnt ? k0 + k : k0) * stride;
#pragma unroll
            for (int hh = 0; hh < kH; ++hh) {
                const int h_loc = h0 + (hh < nh ? hh : 0);
                ml[k][hh] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (slot * p.qh + h_loc) * 2));
                const float *src = p.part_o + (slot * p.qh + h_loc) * D + lane * kPer;
                if constexpr (kPer == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    ov[k][hh][0] = t.x; ov[k][hh][1] = t.y; ov[k][hh][2] = t.z; ov[k][hh][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    ov[k][hh][0] = t.x; ov[k][hh][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int hh = 0; hh < kH; ++hh) {
                if (k0 + k >= cnt || ml[k][hh].x == -INFINITY) continue;
                const float Mn = fmaxf(M[hh], ml[k][hh].x);
                const float a = fast_exp2(M[hh] - Mn), b = fast_exp2(ml[k][hh].x - Mn);
                L[hh] = L[hh] * a + ml[k][hh].y * b;
#pragma unroll
                for (int u = 0; u < kPer; ++u) acc[hh][u] = acc[hh][u] * a + ov[k][hh][u] * b;
                M[hh] = Mn;
            }
    }
    __syncwarp();   // every lane's loads of the children precede the first child's overwrite
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
        if (hh >= nh) break;
        if (dst) {
            const float inv = 1.f / L[hh];
#pragma unroll
            for (int u = 0; u < kPer; u += 2)
                *reinterpret_cast<uint32_t *>(dst + hh * D + lane * kPer + u) =
                    pack_bf16x2(acc[hh][u] * inv, acc[hh][u + 1] * inv);
        } else {
            float *o = p.part_o + (slot0 * p.qh + h0 + hh) * D + lane * kPer;
            if constexpr (kPer == 4) {
                *reinterpret_cast<float4 *>(o) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
            } else {
                *reinterpret_cast<float2 *>(o) = make_float2(acc[hh][0], acc[hh][1]);
            }
            if (lane == 0) *reinterpret_cast<float2 *>(p.part_ml + (slot0 * p.qh + h0 + hh) * 2) = make_float2(M[hh], L[hh]);
        }
    }
}

// ------------------------------------------------------------------ early prefetch
// While the decode CTA waits for the plan, it finds the first units of its
// own slice from context_lens and the block tables (the same partition the
// plan builds: the units of all sequences in order, cut into P equal slices)
// and prefetches their blocks' rows into L2, so the first copies after the wait hit L2.  A
// prefetch is only a hint: it reads inputs before the wait, and a stale value
// would cost time, never a wrong result.  Threads [0, nthr) take part (the
// consumer warps: the producer goes straight on to its wait and first
// copies); they meet at named barrier 1.  warp_tot is shared memory for one
// int per warp.
template <int D>
__device__ __forceinline__ void prefetch_first_blocks(const DecodeParams &p, int nblocks, int32_t *warp_tot,
                                                      int nthr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.num_seqs;
    const int B = 1 << p.log2b;
    const int64_t max_tok = (int64_t)p.max_blocks * B;
    // 1. blocks of this thread's contiguous range of sequences
    const int s0 = (int)((int64_t)S * tid / nthr), s1 = (int)((int64_t)S * (tid + 1) / nthr);
    int sum = 0;
    for (int s = s0; s < s1; s += 8) {          // eight loads in flight at a time
        int c[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) c[u] = s + u < s1 ? __ldg(p.context_lens + s + u) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c[u] >= 1 && c[u] <= max_tok) sum += (c[u] + kU - 1) / kU;
    }
    // 2. exclusive prefix over the threads' ranges
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
    int before = 0, T = 0;
    for (int w = 0; w < nthr / 32; ++w) {
        const int t = warp_tot[w];
        if (w < warp) before += t;
        T += t;
    }
    const int excl = before + incl - sum;
    if (T <= 0 || sum == 0) return;
    // 3. the slice's first nblocks entries: the thread whose range holds one walks to it
    const int64_t NV = (int64_t)T * p.nhg, P = gridDim.x;
    const int64_t lo = (int64_t)blockIdx.x * NV / P, hi = ((int64_t)blockIdx.x + 1) * NV / P;
    const int64_t row_bytes = (int64_t)p.num_kv_heads * D * 2;       // one token of all kv-heads
    const uint32_t span = (uint32_t)(p.kvh * D * 2);                 // the kv-heads of one group
    for (int k = 0; k < nblocks; ++k) {
        const int64_t v = lo + k;
        if (v >= hi) break;
        const int hg = (int)(v / T);
        const int b = (int)(v - (int64_t)hg * T);
        if (b < excl || b >= excl + sum) continue;
        int acc = excl;
        for (int s = s0; s < s1; ++s) {
            const int ctx = __ldg(p.context_lens + s);
            const int nb = (ctx >= 1 && ctx <= max_tok) ? (ctx + kU - 1) / kU : 0;
            if (b < acc + nb) {
                const int u = b - acc;   // the unit, and its rows of its block(s)
                const int32_t *row = p.block_tables + (int64_t)s * p.max_blocks;
                auto pf = [&](int32_t blk, int row0, int nrows) {
                    if (blk < 0 || blk >= p.num_blocks) return;
                    const int64_t base = ((int64_t)blk * B + row0) * row_bytes;
                    if (p.nhg == 1) {
                        prefetch_l2_bulk(p.k_bytes + base, (uint32_t)(nrows * row_bytes));
                        prefetch_l2_bulk(p.v_bytes + base, (uint32_t)(nrows * row_bytes));
                    } else {
                        const int64_t off = base + (int64_t)hg * span;
                        for (int t = 0; t < nrows; ++t) {
                            prefetch_l2_bulk(p.k_bytes + off + t * row_bytes, span);
                            prefetch_l2_bulk(p.v_bytes + off + t * row_bytes, span);
                        }
                    }
                };
                if (p.log2b == 4) {
                    pf(__ldg(row + u), 0, kU);
                } else if (p.log2b == 5) {
                    pf(__ldg(row + (u >> 1)), (u & 1) * kU, kU);
                } else {
                    pf(__ldg(row + 2 * u), 0, 8);
                    if ((2 * u + 1) * 8 < ctx) pf(__ldg(row + 2 * u + 1), 0, 8);
                }
                break;
            }
            acc += nb;
        }
    }
}

// ------------------------------------------------------------------ main kernel
// kTwo: the cache block size is 8, and a unit's K (and V) tile is two 8-row
// TMA boxes, [box][kv-head][D/64 plane][8 rows][64], the second box kv_tile/2
// bytes after the first; otherwise one 16-row box, [kv-head][plane][16 rows][64].
template <int D, bool kTwo>
__global__ void __launch_bounds__(32 * (kMaxConsumerWarps + 1), 1)
    split_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    constexpr int kHeadTileBytes = kU * D * 2;    // one kv-head of one unit
    constexpr int kBoxRows = kTwo ? 8 : kU;       // token rows of one TMA box
    constexpr int kKSteps = D / 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int kvh = p.kvh, NS = p.num_stages;
    const int cwarps = kvh * p.wpk;   // consumer warps; the producer is the next one
    const int kv_tile = kvh * kHeadTileBytes;
    const int q_tile = p.qh * D * 2;
    const int stage_bytes = (2 * kv_tile + q_tile + 1023) & ~1023;
    StageHeader *hdr = reinterpret_cast<StageHeader *>(smem + NS * stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(hdr + NS);
    uint64_t *empty = full + NS;
    __shared__ int abort_flag;
    __shared__ int32_t pf_warp_tot[kMaxConsumerWarps + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, cwarps);
        }
        abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (p.context_lens && warp < cwarps) prefetch_first_blocks<D>(p, NS, pf_warp_tot, 32 * cwarps);
    grid_dependency_wait();      // the plan (and everything before it) is complete
    grid_dependents_launch();    // the next kernel may become resident

    const int S = p.num_seqs;
    const int64_t T = __ldg(p.prefix + S);
    const int64_t NV = T * p.nhg;
    const int64_t P = p.shared_sms ? min((int64_t)gridDim.x, (int64_t)__ldg(p.active)) : (int64_t)gridDim.x;
    if ((int64_t)blockIdx.x >= P) return;   // this SM is left to the prefill kernel
    const int64_t lo = cta_slice_begin(blockIdx.x, NV, P);
    const int64_t hi = cta_slice_begin(blockIdx.x + 1, NV, P);
    const int nloc = (int)(hi - lo);
    if (nloc <= 0) return;

    if (warp == cwarps) {
        // ================= producer warp
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
        auto load_entry = [&](int64_t v, StreamEntry &e, int &hg, int &b1) {
            b1 = -1;
            if (v < hi) {
                hg = (int)(v / T);
                e = p.stream[v - (int64_t)hg * T];
                if (kTwo) b1 = p.stream_b1[v - (int64_t)hg * T];
            } else {
                hg = -1;
                e.seq = -1; e.qrow = 0; e.blk = -1; e.packed = 0;
            }
        };
        StreamEntry cur, nxt;
        int cur_hg, nxt_hg, cur_b1, nxt_b1;
        load_entry(lo + lane, cur, cur_hg, cur_b1);
        int prev_seq = -1, prev_hg = -1;
        int issued = 0;
        bool ok = true;
        for (int64_t base = lo; base < hi && ok; base += 32) {
            load_entry(base + 32 + lane, nxt, nxt_hg, nxt_b1);  // prefetch the next chunk
            const int n = (int)(hi - base < 32 ? hi - base : 32);
            const int next_seq_first = __shfl_sync(0xffffffffu, nxt.seq, 0);
            const int next_hg_first = __shfl_sync(0xffffffffu, nxt_hg, 0);
            for (int i = 0; i < n; ++i) {
                const int seq = __shfl_sync(0xffffffffu, cur.seq, i);
                const int qrow = __shfl_sync(0xffffffffu, cur.qrow, i);
                const int blk = __shfl_sync(0xffffffffu, cur.blk, i);
                const int packed = __shfl_sync(0xffffffffu, cur.packed, i);
                const int hg = __shfl_sync(0xffffffffu, cur_hg, i);
                const int blk1 = kTwo ? __shfl_sync(0xffffffffu, cur_b1, i) : -1;
                const int nseq = i + 1 < 32 ? __shfl_sync(0xffffffffu, cur.seq, (i + 1) & 31) : next_seq_first;
                const int nhg = i + 1 < 32 ? __shfl_sync(0xffffffffu, cur_hg, (i + 1) & 31) : next_hg_first;
                if (lane == 0) {
                    const int k = issued;
                    const int stage = k % NS;
                    if (p.stall == PA_STALL_PRODUCER && k >= p.stall_after) {
                        ok = false;   // test hook: stage k and later are never filled
                    } else if (k >= NS && !mbar_wait(empty + stage, ((k / NS) - 1) & 1, p.wait_ns)) {
                        set_status(p.status, PA_ERR_TIMEOUT);
                        note_wait_site(p.wait_sites, PA_WAIT_DECODE_PRODUCER);
                        abort_flag = 1;
                        ok = false;
                    }
                    if (ok) {
                        const bool first = (seq != prev_seq) || (hg != prev_hg);
                        const bool last = (base + i + 1 == hi) || (nseq != seq) || (nhg != hg);
                        StageHeader h;
                        h.seq = seq;
                        h.qrow = qrow;
                        h.hg = hg;
                        h.lb = packed >> 8;
                        h.ntok = packed & 63;
                        h.flags = (first ? kFirst : 0) | (last ? kLast : 0) |
                                  ((packed >> 6) & 1 ? kSeqEnd : 0) | (blk >= 0 ? kValid : 0);
                        h.pad0 = h.pad1 = 0;
                        hdr[stage] = h;
                        uint8_t *st = smem + (size_t)stage * stage_bytes;
                        const uint32_t bytes = (blk >= 0 ? 2u * kv_tile : 0u) + (first ? (uint32_t)q_tile : 0u);
                        if (bytes) mbar_arrive_expect_tx(full + stage, bytes);
                        else mbar_arrive(full + stage);
                        if (blk >= 0) {
                            const int h0 = hg * kvh;
                            for (int t = 0; t < kvh; t += p.tma_heads) {
                                if (kTwo) {
                                    // two 8-token blocks; past the sequence end the coordinate
                                    // num_blocks is out of bounds and TMA fills zeros
                                    const int b1 = blk1 >= 0 ? blk1 : p.num_blocks;
                                    const int ho = t * (8 * D * 2);
                                    tma_load_5d(st + ho, &tmap_k, 0, 0, 0, h0 + t, blk, full + stage);
                                    tma_load_5d(st + kv_tile / 2 + ho, &tmap_k, 0, 0, 0, h0 + t, b1, full + stage);
                                    tma_load_5d(st + kv_tile + ho, &tmap_v, 0, 0, 0, h0 + t, blk, full + stage);
                                    tma_load_5d(st + kv_tile + kv_tile / 2 + ho, &tmap_v, 0, 0, 0, h0 + t, b1,
                                                full + stage);
                                } else {
                                    // 16 tokens from token tok0 of the block (B = 32: its upper half)
                                    const int tok0 = ((packed >> 7) & 1) * kU;
                                    tma_load_5d(st + t * kHeadTileBytes, &tmap_k, 0, tok0, 0, h0 + t, blk,
                                                full + stage);
                                    tma_load_5d(st + kv_tile + t * kHeadTileBytes, &tmap_v, 0, tok0, 0, h0 + t, blk,
                                                full + stage);
                                }
                            }
                        }
                        if (first) {
                            const __nv_bfloat16 *qsrc =
                                p.q + ((int64_t)qrow * p.num_heads + (int64_t)hg * p.qh) * D;
                            bulk_g2s(st + 2 * kv_tile, qsrc, q_tile, full + stage);
                        }
                        prev_seq = seq;
                        prev_hg = hg;
                        ++issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
            cur = nxt;
            cur_hg = nxt_hg;
            cur_b1 = nxt_b1;
        }
        // wait (bounded, always at the default limit) until every copy this CTA
        // issued has landed
        if (lane == 0) {
            const int first_k = issued > NS ? issued - NS : 0;
            for (int k = first_k; k < issued; ++k) mbar_wait(full + (k % NS), (k / NS) & 1);
        }
        return;
    }

    // ================= consumer warp w: q-heads [hoff, hoff + gcount) of kv-head kh
    // Products taken transposed, so that the 16 tokens of a unit fill the M
    // of m16n8k16 and up to 8 q-heads its N:
    //   S^T (16 tokens x heads) = K Q^T and O^T (D x heads) += V^T P^T.
    // Lane l holds heads 2(l%4) and 2(l%4)+1 (n) of tokens / dims l/4 and
    // l/4+8 (m); the A operands are K (ldmatrix) and V^T (ldmatrix.trans), the
    // B operands Q^T (registers, per sequence) and P^T (S^T's accumulators
    // transposed by movmatrix).  A kv-head with more than 8 q-heads has several
    // warps, each reading the same K/V tile.
    const int kh = warp / p.wpk;
    const int hoff = (warp - kh * p.wpk) * p.gw;
    const int G = p.group;
    const int gcount = min(p.gw, G - hoff);
    const int r = lane >> 2;        // token / dim row of the m16 fragments
    const int quad = lane & 3;      // head columns 2*quad, 2*quad+1
    const bool row_ok = r < gcount; // Q^T column r of the B fragments
    const int h_first = kh * G + hoff;   // this warp's first q-head within the CTA's group
    // ldmatrix lane addressing inside one kv-head tile (128-byte rows, swizzled)
    const int mi = lane >> 3, rr = lane & 7;
    const int k_tok = ((mi >> 1) << 3) + rr, k_dsub = mi & 1;
    const int v_tok = ((mi & 1) << 3) + rr, v_dsub = mi >> 1;
    constexpr int kMTiles = D / 16;

    int k = 0;
    while (k < nloc) {
        // ---- one piece: the blocks of one sequence (and kv-head group) in this slice;
        // its accumulators live only here, so the piece's end has registers to spare
        float ot[kMTiles][4];
        uint32_t qb[kKSteps][2];
        float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < kMTiles; ++j) ot[j][0] = ot[j][1] = ot[j][2] = ot[j][3] = 0.f;
        StageHeader h;
        int piece_lb0 = 0;
        bool aborted = false;
        for (bool first_block = true;; first_block = false) {
            const int stage = k % NS;
            // (another warp may set the flag meanwhile: one answer for the whole warp)
            if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(&abort_flag) != 0)) { aborted = true; break; }
            // test hook: stop without releasing stage k, so the producer's wait runs out
            if (p.stall == PA_STALL_CONSUMER && k >= p.stall_after) { aborted = true; break; }
            if (!mbar_wait_warp(full + stage, (k / NS) & 1, p.wait_ns)) {
                if (lane == 0) {
                    set_status(p.status, PA_ERR_TIMEOUT);
                    note_wait_site(p.wait_sites, PA_WAIT_DECODE_CONSUMER);
                }
                abort_flag = 1;
                aborted = true;
                break;
            }
            h = hdr[stage];
            const uint8_t *st = smem + (size_t)stage * stage_bytes;
            if (first_block) {
                const uint8_t *qs = st + 2 * kv_tile + (size_t)(h_first + r) * D * 2;
#pragma unroll
                for (int ks = 0; ks < kKSteps; ++ks) {
                    qb[ks][0] = row_ok ? *reinterpret_cast<const uint32_t *>(qs + (ks * 16 + quad * 2) * 2) : 0u;
                    qb[ks][1] = row_ok ? *reinterpret_cast<const uint32_t *>(qs + (ks * 16 + 8 + quad * 2) * 2) : 0u;
                }
                piece_lb0 = h.lb;
            }
            if (h.flags & kValid) {
                // byte address of token row t (0..15), 64-column plane pl, of this
                // warp's kv-head in the K (or V) tile at `tile`
                const uint32_t ktile = smem_u32(st), vtile = ktile + kv_tile;
                auto row_addr = [&](uint32_t tile, int pl, int t) -> uint32_t {
                    if (kTwo)
                        return tile + (t >> 3) * (kv_tile >> 1) + kh * (8 * D * 2) + pl * (8 * 128) + (t & 7) * 128;
                    return tile + kh * kHeadTileBytes + pl * (kBoxRows * 128) + t * 128;
                };
                // ---- S^T = K Q^T: A = K (tokens x 16 dims per step), B = Q^T
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < kKSteps; ++ks) {
                    const int chunk = ((ks & 3) << 1) + v_dsub;
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(row_addr(ktile, ks >> 2, v_tok) + ((chunk ^ (v_tok & 7)) << 4), a0, a1, a2, a3);
                    mma_bf16_16816(s4, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
                // ---- online softmax per head column (heads 2q, 2q+1; tokens r, r+8)
                const int ntok = h.ntok;
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = (r + (i >> 1) * 8) < ntok ? s4[i] * p.scale_log2 : -INFINITY;
                float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                // ntok >= 1, so every column has a finite max
                const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                const float al0 = fast_exp2(m_run[0] - mn0), al1 = fast_exp2(m_run[1] - mn1);
                const float p0 = fast_exp2(x[0] - mn0), p1 = fast_exp2(x[1] - mn1);
                const float p2 = fast_exp2(x[2] - mn0), p3 = fast_exp2(x[3] - mn1);
                l_part[0] = l_part[0] * al0 + (p0 + p2);
                l_part[1] = l_part[1] * al1 + (p1 + p3);
                m_run[0] = mn0;
                m_run[1] = mn1;
#pragma unroll
                for (int j = 0; j < kMTiles; ++j) {
                    ot[j][0] *= al0;
                    ot[j][1] *= al1;
                    ot[j][2] *= al0;
                    ot[j][3] *= al1;
                }
                // P^T as the B operand: (token, head) pairs transposed to (head, token)
                const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));   // tokens 0..7
                const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));   // tokens 8..15
                // masks for value rows past the sequence end (they may hold anything)
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (ntok < kU) {
                    const int t0 = quad * 2;
                    mlo = (t0 < ntok ? 0x0000ffffu : 0u) | (t0 + 1 < ntok ? 0xffff0000u : 0u);
                    mhi = (t0 + 8 < ntok ? 0x0000ffffu : 0u) | (t0 + 9 < ntok ? 0xffff0000u : 0u);
                }
                // ---- O^T += V^T P^T: A = V^T (16 dims x 16 tokens per m-tile)
#pragma unroll
                for (int j = 0; j < kMTiles; ++j) {
                    const int chunk = ((j & 3) << 1) + k_dsub;
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(row_addr(vtile, j >> 2, k_tok) + ((chunk ^ (k_tok & 7)) << 4), v0, v1, v2, v3);
                    v0 &= mlo; v1 &= mlo; v2 &= mhi; v3 &= mhi;
                    mma_bf16_16816(ot[j], v0, v1, v2, v3, pb0, pb1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + stage);
            ++k;
            if ((h.flags & kLast) || k >= nloc) break;
        }
        if (aborted) break;

        // ---- the piece's end
        float l0 = l_part[0], l1 = l_part[1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const bool whole = piece_lb0 == 0 && (h.flags & kSeqEnd);
        const int64_t out_row = (int64_t)h.qrow * p.num_heads + (int64_t)h.hg * p.qh;
        const int64_t vs = (int64_t)h.hg * S + h.seq;
        const int64_t slot = vs + blockIdx.x;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int hh = 2 * quad + e;
            if (hh >= gcount) continue;
            const int h_loc = h_first + hh;
            const float l_e = e ? l1 : l0;
            if (whole) {
                const float inv = 1.f / l_e;
                __nv_bfloat16 *dst = p.out + (out_row + h_loc) * D + r;
#pragma unroll
                for (int j = 0; j < kMTiles; ++j) {
                    dst[j * 16] = __float2bfloat16_rn(ot[j][e] * inv);
                    dst[j * 16 + 8] = __float2bfloat16_rn(ot[j][2 + e] * inv);
                }
            } else {
                float *dst = p.part_o + (slot * p.qh + h_loc) * D + r;
#pragma unroll
                for (int j = 0; j < kMTiles; ++j) {
                    dst[j * 16] = ot[j][e];
                    dst[j * 16 + 8] = ot[j][2 + e];
                }
                if (r == 0)
                    *reinterpret_cast<float2 *>(p.part_ml + (slot * p.qh + h_loc) * 2) = make_float2(m_run[e], l_e);
            }
        }
        if (whole) continue;
        // a piece of a sequence cut by CTA boundaries, now stored: count it in;
        // the warp that stores the last of the sequence's pieces merges them
        // (the stream's sizes are reloaded here rather than kept in registers)
        const int64_t Tt = __ldg(p.prefix + S);
        const int64_t NVt = Tt * p.nhg;
        const int64_t Pt = p.shared_sms ? min((int64_t)gridDim.x, (int64_t)__ldg(p.active)) : (int64_t)gridDim.x;
        const int64_t b0 = __ldg(p.prefix + h.seq), b1 = __ldg(p.prefix + h.seq + 1);
        const int64_t c0 = cta_of(h.hg * Tt + b0, NVt, Pt), c1 = cta_of(h.hg * Tt + b1 - 1, NVt, Pt);
        int pieces = (int)(c1 - c0 + 1);
        if (NVt >= Pt && pieces >= kTreeMinPieces) {
            // many pieces (no slice is empty here): group by group, up the sequence's tree
            int node = (int)((int64_t)blockIdx.x - c0);
            bool last = true;
            int base = 0;   // groups at the levels below
            for (int l = 0; (1 << (2 * l)) < pieces; ++l) {
                const int child = 1 << (2 * l), span = child * kTreeFan;
                const int g = node / span, first = g * span;
                const int cnt = min(kTreeFan, (pieces - first + child - 1) / child);
                if (cnt >= 2) {
                    __syncwarp();   // every lane's stores precede lane 0's release
                    int got = 0;
                    if (lane == 0) got = atomic_add_acq_rel_gpu(p.arrivals + (c0 + base + g) * kMaxConsumerWarps + warp, 1);
                    last = __shfl_sync(0xffffffffu, got, 0) == cnt - 1;   // (orders the acquire before the loads)
                    if (!last) break;   // a later child merges the group
                    const bool root = span >= pieces;
                    for (int h = 0; h < gcount; h += 4)
                        merge_group<D>(p, vs + c0 + first, child, cnt, h_first + h, gcount - h < 4 ? gcount - h : 4,
                                       root ? p.out + (out_row + h_first + h) * D : nullptr);
                    if (root) break;
                }
                node = first;
                base += tree_groups(l, pieces);
            }
            continue;
        }
        if (NVt < Pt) {
            pieces = 0;
            for (int64_t c = c0; c <= c1; ++c)
                pieces += cta_slice_begin(c, NVt, Pt) < cta_slice_begin(c + 1, NVt, Pt) ? 1 : 0;
        }
        __syncwarp();   // every lane's stores precede lane 0's release
        int merge = 0;
        if (lane == 0) merge = atomic_add_acq_rel_gpu(p.arrivals + c0 * kMaxConsumerWarps + warp, 1) == pieces - 1;
        merge = __shfl_sync(0xffffffffu, merge, 0);   // (also orders lane 0's acquire before the loads)
        if (merge) {
            for (int g = 0; g < gcount; g += 4)
                merge_pieces<D>(p, vs, c0, c1, NVt, Pt, h_first + g, gcount - g < 4 ? gcount - g : 4,
                                p.out + (out_row + h_first + g) * D);
        }
    }
}

// ------------------------------------------------------------------ host side
// Pool [num_blocks][B][Hkv][D] bf16 seen as a 5-D tensor whose box is
// min(B, 16) tokens of one block for `box_heads` kv-heads, laid out in shared
// memory as [head][D/64][token][64] with 128-byte rows and the 128-byte swizzle.
CUresult make_pool_map(CUtensorMap *map, const void *pool, int num_blocks, int B, int hkv, int D,
                       int box_heads, bool permuted) {
    auto encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t eb = 2;
    cuuint64_t dims[5];
    cuuint64_t strides[4];
    cuuint32_t box[5];
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (permuted) {
        // dims: d_lo(64), token(B), d_hi(D/64), head(Hkv), block
        dims[0] = 64; dims[1] = B; dims[2] = D / 64; dims[3] = hkv; dims[4] = num_blocks;
        strides[0] = (cuuint64_t)hkv * D * eb;   // token
        strides[1] = 64 * eb;                     // d_hi
        strides[2] = (cuuint64_t)D * eb;          // head
        strides[3] = (cuuint64_t)B * hkv * D * eb;   // block
        box[0] = 64; box[1] = B < kU ? B : kU; box[2] = D / 64; box[3] = box_heads; box[4] = 1;
    } else {
        return CUDA_ERROR_INVALID_VALUE;
    }
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

struct Layout {
    int kvh, wpk, gw, group, qh, nhg;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory stages of the ring (up to 8) for one 16-token unit of kvh
// kv-heads and the CTA's qh query heads.
int stages_for(int kvh, int qh, int D) {
    const int kv_tile = kvh * kU * D * 2;
    const int stage_bytes = (int)align_up(2 * kv_tile + qh * D * 2, 1024);
    int ns = (kSmemBudget - 1024) / (stage_bytes + (int)sizeof(StageHeader) + 16);
    return ns > 8 ? 8 : ns;
}

// kv-heads per CTA: up to 8 consumer warps of at most 8 q-heads each and up to
// 32 q-heads in all, dividing the kv-heads evenly, and few enough that a unit
// leaves room for three stages.
Layout decode_layout(int num_heads, int num_kv_heads, int D) {
    Layout L;
    L.group = num_heads / num_kv_heads;
    L.wpk = (L.group + kHeadsPerWarp - 1) / kHeadsPerWarp;
    L.gw = (L.group + L.wpk - 1) / L.wpk;
    int kvh = kMaxConsumerWarps / L.wpk;
    if (kvh > kMaxKvhPerCta) kvh = kMaxKvhPerCta;
    if (kvh > num_kv_heads) kvh = num_kv_heads;
    while (kvh > 1 && (kvh * L.group > kMaxQHeadsPerCta || num_kv_heads % kvh != 0 ||
                       stages_for(kvh, kvh * L.group, D) < 3))
        --kvh;
    L.kvh = kvh;
    L.qh = kvh * L.group;
    L.nhg = num_kv_heads / kvh;
    return L;
}

// 16-token units of a sequence of max_blocks blocks of B tokens.
int64_t max_units(int max_blocks, int B) { return ((int64_t)max_blocks * B + kU - 1) / kU; }

// Workspace: the plan's prefix [S + 1] and SM split, the arrival counters of
// cut sequences [kPartialCtas][kMaxConsumerWarps], the unit stream
// [S * max units] (B = 8: and its second blocks), then the partials,
// slot = hg*S + s + CTA (< NHG*S + CTAs): (m, l) [slots][QH][2] and
// o [slots][QH][D], fp32.
struct WorkspaceLayout {
    size_t prefix, active, arrivals, stream, stream_b1, part_ml, part_o, total;
};

WorkspaceLayout workspace_layout(int num_seqs, int num_heads, int head_dim, int max_blocks, int B) {
    WorkspaceLayout w;
    const size_t slots_heads = ((size_t)num_seqs + kPartialCtas) * num_heads;
    const size_t units = (size_t)num_seqs * (size_t)max_units(max_blocks, B);
    w.prefix = 0;
    w.active = align_up(sizeof(int32_t) * ((size_t)num_seqs + 1), 16);
    w.arrivals = align_up(w.active + sizeof(int32_t), 256);
    w.stream = align_up(w.arrivals + sizeof(int32_t) * kPartialCtas * kMaxConsumerWarps, 256);
    w.stream_b1 = align_up(w.stream + sizeof(StreamEntry) * units, 256);
    w.part_ml = align_up(w.stream_b1 + (B < kU ? sizeof(int32_t) * units : 0), 256);
    w.part_o = align_up(w.part_ml + sizeof(float) * 2 * slots_heads, 256);
    w.total = align_up(w.part_o + sizeof(float) * (size_t)head_dim * slots_heads, 256);
    return w;
}

template <int D, bool kTwo>
cudaError_t launch_main(const DecodeParams &prm, const CUtensorMap &mk, const CUtensorMap &mv,
                        int grid, cudaStream_t stream, bool timed) {
    const int kv_tile = prm.kvh * kU * D * 2;
    const int stage_bytes = (int)align_up(2 * kv_tile + prm.qh * D * 2, 1024);
    const size_t smem = 1024 + (size_t)prm.num_stages * (stage_bytes + sizeof(StageHeader) + 16);
    auto kern = split_decode_kernel<D, kTwo>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (timed) timing_begin(stream);
    e = launch_dependent(kern, dim3(grid), dim3(32 * (prm.kvh * prm.wpk + 1)), smem, stream, mk, mv, prm);
    if (timed) timing_end(stream);
    return e;
}

int log2_of_block(int B) { return B == 8 ? 3 : (B == 16 ? 4 : (B == 32 ? 5 : -1)); }

}  // namespace

bool split_decode_supported(const AttnArgs &a) {
    if (a.dtype != PA_DTYPE_BF16 || log2_of_block(a.block_size) < 0) return false;
    if (a.head_dim != 64 && a.head_dim != 128) return false;
    if (a.num_seqs > kMaxSeqs) return false;
    // a stream entry holds unit << 8: units of a sequence stay below 2^23
    if (max_units(a.max_blocks, a.block_size) >= (int64_t)1 << 23) return false;
    if ((int64_t)a.num_seqs * max_units(a.max_blocks, a.block_size) >= (int64_t)1 << 30) return false;
    const int G = a.num_heads / a.num_kv_heads;
    if (G > kMaxGroup) return false;
    const Layout L = decode_layout(a.num_heads, a.num_kv_heads, a.head_dim);
    if (L.qh > kMaxQHeadsPerCta) return false;
    if (stages_for(L.kvh, L.qh, a.head_dim) < 2) return false;
    auto al = [](const void *ptr, uintptr_t n) { return reinterpret_cast<uintptr_t>(ptr) % n == 0; };
    return al(a.q, 16) && al(a.k_cache, 16) && al(a.v_cache, 16) && al(a.out, 4);
}

size_t split_decode_workspace(int num_seqs, int num_heads, int head_dim, int max_blocks, int block_size) {
    return workspace_layout(num_seqs, num_heads, head_dim, max_blocks, block_size).total;
}

cudaError_t launch_split_decode(const AttnArgs &a, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream, bool timed, const KvWriteArgs *write,
                                const PrefillPlanJob *prefill,
                                const std::function<cudaError_t()> *between) {
    const bool share_sms = prefill != nullptr;
    if (a.num_seqs == 0) return cudaSuccess;
    const int B = a.block_size;
    const WorkspaceLayout w = workspace_layout(a.num_seqs, a.num_heads, a.head_dim, a.max_blocks, B);
    if (workspace_bytes < w.total) return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const Layout L = decode_layout(a.num_heads, a.num_kv_heads, a.head_dim);

    DecodeParams prm;
    prm.q = static_cast<const __nv_bfloat16 *>(a.q);
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.prefix = reinterpret_cast<const int32_t *>(ws + w.prefix);
    prm.stream = reinterpret_cast<const StreamEntry *>(ws + w.stream);
    prm.stream_b1 = reinterpret_cast<const int32_t *>(ws + w.stream_b1);
    prm.log2b = log2_of_block(B);
    prm.part_ml = reinterpret_cast<float *>(ws + w.part_ml);
    prm.part_o = reinterpret_cast<float *>(ws + w.part_o);
    prm.num_seqs = a.num_seqs;
    prm.num_heads = a.num_heads;
    prm.kvh = L.kvh;
    prm.wpk = L.wpk;
    prm.gw = L.gw;
    prm.group = L.group;
    prm.qh = L.qh;
    prm.nhg = L.nhg;
    prm.active = reinterpret_cast<const int32_t *>(ws + w.active);
    prm.arrivals = reinterpret_cast<int32_t *>(ws + w.arrivals);
    prm.shared_sms = prefill ? 1 : 0;
    prm.num_stages = stages_for(L.kvh, L.qh, a.head_dim);
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    prm.status = a.status;
    // decode calls (one query row per sequence, all CTAs take a slice): each
    // CTA prefetches its first blocks into L2 while it waits for the plan
    const bool early = !share_sms && a.cu_seqlens_q == nullptr && a.num_seqs <= kMaxSeqsEarlyPrefetch;
    prm.context_lens = early ? a.context_lens : nullptr;
    prm.block_tables = a.block_tables;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.num_kv_heads = a.num_kv_heads;
    prm.k_bytes = static_cast<const uint8_t *>(a.k_cache);
    prm.v_bytes = static_cast<const uint8_t *>(a.v_cache);
    const WaitTest &wt = wait_test();
    prm.wait_ns = wt.limit_ns;
    prm.stall = wt.stall;
    prm.stall_after = wt.after;
    prm.wait_sites = wt.sites;

    // tensor maps: one TMA per unit (two at B = 8) for all kv-heads of the CTA
    CUtensorMap mk, mv;
    prm.tma_heads = L.kvh;
    if (make_pool_map(&mk, a.k_cache, a.num_blocks, B, a.num_kv_heads, a.head_dim, L.kvh, true) != CUDA_SUCCESS ||
        make_pool_map(&mv, a.v_cache, a.num_blocks, B, a.num_kv_heads, a.head_dim, L.kvh, true) != CUDA_SUCCESS) {
        // one TMA per kv-head
        prm.tma_heads = 1;
        if (make_pool_map(&mk, a.k_cache, a.num_blocks, B, a.num_kv_heads, a.head_dim, 1, true) != CUDA_SUCCESS ||
            make_pool_map(&mv, a.v_cache, a.num_blocks, B, a.num_kv_heads, a.head_dim, 1, true) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }

    KvWriteJob job = {};
    if (write) {
        job.seq_start = write->seq_start;
        job.cu_new = write->cu_seqlens_new;
        job.total_new = write->total_new;
        job.key = static_cast<const uint4 *>(write->key);
        job.value = static_cast<const uint4 *>(write->value);
        job.key_stride_v = write->key_stride_tok * 2 / 16;
        job.value_stride_v = write->value_stride_tok * 2 / 16;
        job.k_cache = static_cast<uint4 *>(const_cast<void *>(a.k_cache));
        job.v_cache = static_cast<uint4 *>(const_cast<void *>(a.v_cache));
        job.slot_mapping = write->slot_mapping;
        job.row_vecs = a.num_kv_heads * a.head_dim * 2 / 16;
        job.pool_slots = (int64_t)a.num_blocks * B;
    }

    // plan (and the folded cache write)
    size_t plan_smem = sizeof(int32_t) * ((size_t)a.num_seqs + 1);
    if (share_sms && plan_smem < (size_t)kPrefillPlanSmem) plan_smem = kPrefillPlanSmem;
    auto plan_kern = share_sms ? decode_plan_kernel<true> : decode_plan_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(plan_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_smem);
    if (e != cudaSuccess) return e;
    const int64_t max_entries = (int64_t)a.num_seqs * max_units(a.max_blocks, B);
    const int sms = device_sm_count();
    int grid = sms;
    if (grid > kPartialCtas) grid = kPartialCtas;
    DecodeSplit split;
    split.active = reinterpret_cast<int32_t *>(ws + w.active);
    split.arrivals = prm.arrivals;
    split.num_arrivals = grid * kMaxConsumerWarps;
    split.grid = grid;
    split.share = share_sms ? 1 : 0;
    split.causal = a.causal;
    split.block_ns = (double)kU * a.num_kv_heads * a.head_dim * 2 * 2 / kDecodeBytesPerSmNs;
    split.pair_ns = 4.0 * a.num_heads * a.head_dim / kPrefillFlopsPerSmNs;
    int plan_grid = (int)((max_entries + 4 * kPlanThreads - 1) / (4 * kPlanThreads));
    if (plan_grid > 2 * sms) plan_grid = 2 * sms;
    if (plan_grid < 1) plan_grid = 1;
    // write items: a new token's row in chunks of 128 16-byte vectors, one warp each
    const int64_t write_items =
        write ? (int64_t)write->total_new * ((job.row_vecs + 127) / 128) : 0;
    int write_grid = (int)((write_items + kPlanThreads / 32 - 1) / (kPlanThreads / 32));
    if (write_grid > 2 * sms) write_grid = 2 * sms;
    job.first_cta = plan_grid;
    plan_grid += write_grid;                    // + the CTAs of the cache write
    if (share_sms) ++plan_grid;                 // + the CTA that plans the prefill chunks
    const PrefillPlanJob pf = share_sms ? *prefill : PrefillPlanJob{};
    e = launch_dependent(plan_kern, dim3(plan_grid), dim3(kPlanThreads), plan_smem, stream,
                         a.context_lens, a.cu_seqlens_q, a.block_tables, a.num_seqs, a.max_blocks,
                         a.num_blocks, a.total_q, log2_of_block(B), reinterpret_cast<int32_t *>(ws + w.prefix),
                         reinterpret_cast<StreamEntry *>(ws + w.stream), reinterpret_cast<int32_t *>(ws + w.stream_b1),
                         a.status, job, split, pf);
    if (e != cudaSuccess) return e;

    const bool two = B < kU;   // B = 8: two blocks per unit
    if (a.head_dim == 64) e = two ? launch_main<64, true>(prm, mk, mv, grid, stream, timed)
                                  : launch_main<64, false>(prm, mk, mv, grid, stream, timed);
    else e = two ? launch_main<128, true>(prm, mk, mv, grid, stream, timed)
                 : launch_main<128, false>(prm, mk, mv, grid, stream, timed);
    if (e != cudaSuccess) return e;
    return between ? (*between)() : cudaSuccess;
}

}  // namespace pa
