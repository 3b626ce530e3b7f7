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
// 128 (16, 8 or 4 cache blocks); K and V of a tile take one slot each of a TMA
// ring, both with one box per cache block.
// Warp roles: warps 0-7 two softmax warpgroups (thread = row = TMEM lane of
// its tile), warp 8 TMA producer, warp 9 TMEM owner and MMA issuer, warps
// 12-15 the output warpgroup (O / l to the rows of out).
//   S_t = Q_t K_j^T                         -> TMEM, fp32 (128 columns per tile)
//   P_t = exp2(S_t * scale*log2e - m)       -> TMEM over S_t, bf16 pairs, in two halves
//   O_t += P_t V_j                          -> TMEM, fp32; A operand P_t read from TMEM
// The two M-tiles alternate on the tensor pipe: while one softmax warpgroup
// turns S into P, the products of the other tile run; the first half of P
// goes to the tensor pipe while the second is computed.
// The running max is only raised (and O rescaled in TMEM) when a row's max
// grows by more than 2^8; otherwise the stale max is kept, which changes no
// result because l uses the same max.  Causal masking is a select on the
// logits; keys of blocks past the sequence end come in as zeros (TMA
// out-of-bounds fill), and value rows past the context end inside the last
// block are zeroed in shared memory so P * V never sees 0 * NaN.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "prefill_plan.cuh"

namespace pa {
namespace {

constexpr int BM = 128;               // rows per M-tile
constexpr int kMT = 2;                // M-tiles per CTA, one softmax warpgroup each
constexpr int BN = 128;               // keys per KV tile (8 cache blocks)
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kProducerWarp = 4 * kMT;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kOutWarp = kProducerWarp + 4;       // first warp of the output warpgroup
// warpgroups: the softmax ones, the producer / MMA one (two warps idle), the output one
constexpr int kThreads = 32 * (4 * kMT + 8);
// Register split: launched at 128 a thread (512 x 128 = 64K), the producer /
// MMA and the output warpgroups drop to kRegsSide and kRegsOut and the
// softmax warpgroups rise to kRegsSoftmax, within the launch's total.
constexpr int kRegsLaunch = 128;
constexpr int kRegsSide = 56;
constexpr int kRegsOut = 56;
constexpr int kRegsSoftmax = 200;
static_assert(128 * (kRegsSide + kRegsOut) + 128 * kMT * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
constexpr int kPlanThreads = 512;
constexpr int kTmemCols = 512;

struct PrefillParams {
    const int32_t *cu_seqlens_q;
    const int32_t *context_lens;
    const int32_t *block_tables;
    const int2 *entries;       // (sequence, CTA tile), most KV tiles first
    const int32_t *num_entries;
    int32_t *next_item;        // work counter, zeroed by the plan kernel
    __nv_bfloat16 *out;
    int num_seqs;
    int total_q;
    int max_q_len;
    int num_heads;
    int num_kv_heads;
    int group;       // q-heads per kv-head
    int pos_shift;   // log2(query positions per M-tile) = log2(128 / group)
    int max_blocks;
    int num_blocks;
    float scale_log2;
    int32_t *status;
    int causal;      // 0: encode-only, every row sees the whole sequence
    // 1: launched behind the decode kernel of the same batch, whose plan launch
    // also built this kernel's plan.  That plan is complete before the launch
    // (every decode CTA waited for it before this grid could start), so there is
    // no wait at the start; the wait for the decode grid comes at the end, so
    // this grid completes after it and later work may rely on both.
    int wait_at_end;
    // bounded waits: their limit, and the test hook's stall (PA_STALL_*)
    uint64_t wait_ns;
    int stall;
    int stall_after;
    int32_t *wait_sites;
};

static_assert(BN == kPrefillKeysPerTile, "the plan counts KV tiles of the main kernel's width");

// ------------------------------------------------------------------ plan
// One CTA builds the work list (see prefill_plan.cuh).
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const PrefillPlanJob job) {
    extern __shared__ __align__(16) uint8_t plan_smem[];
    // the main kernel may start its prologue now; it waits for this grid
    // before it reads the plan
    grid_dependents_launch();
    prefill_plan_block(job, plan_smem);
}

// ------------------------------------------------------------------ main kernel
template <int D> struct Shape {
    static constexpr int kDH = D / 64;                 // 64-column planes of a head
    static constexpr int kQBytes = BM * D * 2;         // one M-tile of Q
    static constexpr int kSlotBytes = BN * D * 2;      // K or V of one KV tile
    static constexpr int kPlaneQ = BM * 128;           // one 64-column plane of Q
    static constexpr int kBarBytes = 2816;     // barriers, TMEM address, item slots, row sums
    static constexpr int kFit = (int)((kSmemLimit - kMT * kQBytes - kBarBytes) / kSlotBytes);
    static constexpr int kSlots = kFit < 8 ? kFit : 8;  // K/V ring depth
    static constexpr size_t kSmem = (size_t)kMT * kQBytes + (size_t)kSlots * kSlotBytes + kBarBytes;
    static_assert(kSlots >= 3, "the K/V ring needs at least three slots");
    static_assert(kSmem <= kSmemLimit, "shared memory");
};

// One work item: CTA tile `entries[w / Hkv]` of kv-head w % Hkv.  `live` = 0
// marks the end of the work; `valid` = 0 an item the kernel rejects.
struct Item {
    int s, g, q0, q_len, ctx, i0, nrows_all, pos_base, nkv, nb;
    int valid, live;
};
constexpr int kItemSlots = 4;                 // items published ahead of their use

template <int kB>
__device__ __forceinline__ Item decode_item(const PrefillParams &p, int w) {
    Item it;
    const int e = w / p.num_kv_heads;
    it.g = w - e * p.num_kv_heads;
    const int2 ent = p.entries[e];
    it.s = ent.x;
    it.q0 = __ldg(p.cu_seqlens_q + it.s);
    it.q_len = __ldg(p.cu_seqlens_q + it.s + 1) - it.q0;
    it.ctx = __ldg(p.context_lens + it.s);
    const int cta_shift = p.pos_shift + 1;             // kMT = 2 M-tiles per CTA tile
    it.i0 = ent.y << cta_shift;
    it.nrows_all = min(1 << cta_shift, it.q_len - it.i0);
    it.pos_base = it.ctx - it.q_len + it.i0;
    it.nkv = prefill_tile_kv_tiles(it.q_len, it.ctx, ent.y, cta_shift, p.causal);
    it.nb = (it.ctx + kB - 1) / kB;
    it.valid = it.nkv > 0 && (int64_t)it.ctx <= (int64_t)p.max_blocks * kB &&
               it.q_len <= p.max_q_len && it.q0 >= 0 && it.q0 + it.q_len <= p.total_q;
    it.live = 1;
    return it;
}

// Persistent: one CTA per SM takes work items from a counter until none are
// left.  The producer fetches the next item and starts its Q and K/V copies
// while the tensor pipe and the softmax warpgroups still finish the current
// one; the K/V ring, the TMEM buffers and every barrier carry over from item
// to item, their phases counted by running totals that all roles keep alike.
template <int D, int kB>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    constexpr int kBlocksPerTile = BN / kB;          // cache blocks per KV tile
    static_assert(kBlocksPerTile <= 32, "one TMA box per producer lane");
    using SH = Shape<D>;
    constexpr int kDH = SH::kDH, kQBytes = SH::kQBytes, kSlotBytes = SH::kSlotBytes;
    constexpr int kPlaneQ = SH::kPlaneQ, kSlots = SH::kSlots;
    // V tile layout, block-major: [block][D/64 plane][B rows][64], one TMA box
    // per block for all planes.  Key k
    // sits at (k / B) * kVBlockBytes + (k % B) * 128 in a plane; 16-key MMA steps
    // 0..3 of 64 keys start at 0, kVS1, kVS2 and kVS2 + kVS1; their 8-row groups
    // are kVSbo apart and their planes B*128.
    constexpr int kVBlockBytes = kDH * kB * 128;                       // one block, all planes
    constexpr int kVS1 = (16 / kB) * kVBlockBytes + (16 % kB) * 128;
    constexpr int kVS2 = (32 / kB) * kVBlockBytes + (32 % kB) * 128;
    static_assert(((48 / kB) * kVBlockBytes + (48 % kB) * 128) == kVS1 + kVS2, "step 3 = s2 + s1");
    constexpr int kVChunk = 64 / kB * kVBlockBytes;                    // 64 keys
    constexpr int kVLbo = kB * 128;
    constexpr int kVSbo = kB < 16 ? kVBlockBytes : 1024;
    // K tile layout, block-major too, one TMA box per block: a block is
    // [B/8 row group][D/64 plane][8 rows][64], so across the tile the 8-row
    // groups of one plane sit D/64 * 1024 bytes apart (the K-major operand's
    // single group stride) and the planes 1024 bytes apart.
    constexpr int kKSbo = kDH * 1024;
    constexpr int kKPlane = 1024;
    constexpr uint32_t kIdescQK = umma_idesc_bf16(BM, BN, 0);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(BM, D, 1);
    constexpr uint32_t kFull = 0xffffffffu;

    // all shared state is dynamic so the 1024-byte aligned tiles start at 0:
    // Q[2] | K/V ring slots | barriers | item slots
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *q_s = smem;
    uint8_t *kv_s = smem + kMT * kQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(kv_s + kSlots * kSlotBytes);
    uint64_t *q_full = bars;                       // Q of the item landed
    uint64_t *q_empty = q_full + 1;                // every QK product of the item done
    uint64_t *kv_full = q_empty + 1;               // [kSlots]: slot landed
    uint64_t *kv_empty = kv_full + kSlots;         // [kSlots]: slot read by its products
    uint64_t *s_full = kv_empty + kSlots;          // [tile]: S_t written
    uint64_t *p_full = s_full + kMT;               // [tile]: P_t written (and O_t rescaled)
    uint64_t *o_full = p_full + kMT;               // [tile]: last product of the item into O_t done
    uint64_t *p_half = o_full + kMT;               // [tile]: P_t's first 64 keys written (and O_t rescaled)
    uint64_t *o_empty = p_half + kMT;              // [tile]: O_t read by the output warpgroup
    uint64_t *l_full = o_empty + kMT;              // [tile]: the item's row sums of tile t written
    uint64_t *item_full = l_full + kMT;            // [kItemSlots]: item published
    uint64_t *item_empty = item_full + kItemSlots; // [kItemSlots]: item read by every consumer
    uint64_t *drained = item_empty + kItemSlots;   // every product issued has completed
    uint32_t &tmem_base_s = *reinterpret_cast<uint32_t *>(drained + 1);
    Item *items = reinterpret_cast<Item *>(drained + 2);       // [kItemSlots]
    float *l_s = reinterpret_cast<float *>(items + kItemSlots);   // [item parity][tile][row]: row sums
    static_assert((3 + 2 * kSlots + 6 * kMT + 2 * kItemSlots) * 8 + kItemSlots * sizeof(Item) +
                          2 * kMT * BM * sizeof(float) <= SH::kBarBytes,
                  "barrier area");

    // the warp index broadcast from lane 0 is provably warp-uniform, so each
    // role's branch is uniform and the MMA operands stay in uniform registers
    // (computed per lane, a tcgen05.mma issue costs several times its run time)
    const int tid = threadIdx.x, warp = __shfl_sync(kFull, tid >> 5, 0), lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
        if (tid == 0) set_status(p.status, PA_ERR_CUDA);
        if (p.wait_at_end) grid_dependency_wait();
        return;
    }
    const int POS = 1 << p.pos_shift;                  // query positions per M-tile

    if (tid == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(kv_full + i, 1);
            mbar_init(kv_empty + i, 1);
        }
        for (int t = 0; t < kMT; ++t) {
            mbar_init(s_full + t, 1);
            mbar_init(p_full + t, BM);
            mbar_init(o_full + t, 1);
            mbar_init(p_half + t, BM);
            mbar_init(o_empty + t, BM);
            mbar_init(l_full + t, BM);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(item_full + i, 1);
            mbar_init(item_empty + i, 1 + 4 * kMT + 4);  // the MMA warp, every softmax and output warp
        }
        mbar_init(drained, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tmem_alloc(&tmem_base_s, kTmemCols);
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tmap_q);
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // everything above overlaps the plan kernel; the plan (and every earlier
    // write in the stream) is visible after this wait
    if (!p.wait_at_end) grid_dependency_wait();
    const int total = p.num_entries[0] * p.num_kv_heads;   // plain load: written by the plan grid
    const uint32_t tmem = tmem_base_s;
    // TMEM columns: S_t at t*BN (fp32, BN columns); P_t, bf16 pairs, over the
    // first BN/2 columns of S_t; O_t at kMT*BN + t*D
    auto s_col = [](int t) { return (uint32_t)(t * BN); };
    auto o_col = [](int t) { return (uint32_t)(kMT * BN + t * D); };
    // K/V ring: per item, entry n0 + 2j is K of KV tile j, n0 + 2j + 1 its V
    auto slot_of = [](int n) { return n % kSlots; };
    auto phase_of = [](int n) { return (uint32_t)((n / kSlots) & 1); };
    // consumers: item `it` as the producer decoded it, with the read acknowledged
    auto take_item = [&](int it, Item &I) -> bool {
        if (!mbar_wait_warp(item_full + it % kItemSlots, (uint32_t)((it / kItemSlots) & 1), p.wait_ns)) return false;
        I = items[it % kItemSlots];
        __syncwarp();
        if (lane == 0) mbar_arrive(item_empty + it % kItemSlots);
        return true;
    };

    if (warp >= kOutWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOut));
        // ================= output warpgroup: thread r writes row r of M-tile t
        // as O_t / l, after the item's last product into O_t; the MMA warp
        // waits for its o_empty before the next item's first product into O_t
        const int r = tid & (BM - 1);
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        bool ok = true;
        int no = 0;
        for (int it = 0; ok; ++it) {
            Item I;
            if (!take_item(it, I)) { ok = false; break; }
            if (!I.live) break;
            if (!I.valid) continue;
            for (int t = 0; t < kMT; ++t) {
                if (!mbar_wait_warp(o_full + t, (uint32_t)(no & 1), p.wait_ns) ||
                    !mbar_wait_warp(l_full + t, (uint32_t)(no & 1), p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv = 1.f / l_s[((no & 1) * kMT + t) * BM + r];
                const int i = t * POS + (r & (POS - 1));    // position index within the CTA tile
                const bool row_valid = i < I.nrows_all;
                __nv_bfloat16 *dst = p.out + ((int64_t)(I.q0 + I.i0 + (row_valid ? i : 0)) * p.num_heads +
                                              (int64_t)I.g * p.group + (r >> p.pos_shift)) * D;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o0[16], o1[16];
                    tmem_ld16(lane_addr + o_col(t) + 32 * c, o0);
                    tmem_ld16(lane_addr + o_col(t) + 32 * c + 16, o1);
                    tmem_wait_ld();
                    if (c == D / 32 - 1) {       // O_t read: the next item's products may overwrite it
                        tc_fence_before();
                        mbar_arrive(o_empty + t);
                    }
                    if (row_valid) {
                        // 32-byte stores: whole sectors of the row
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t *v = h ? o1 : o0;
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
                            st_global_v8(dst + 32 * c + 16 * h, w);
                        }
                    }
                }
            }
            if (!ok) break;
            ++no;
        }
        if (!ok && r == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            note_wait_site(p.wait_sites, PA_WAIT_PREFILL_SOFTMAX);
        }
    } else if (warp >= kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsSide));
    if (warp == kProducerWarp) {
        // ================= TMA producer
        bool ok = true, stopped = false;
        int n = 0, nq = 0, issued_end = 0;   // issued_end: ring entries issued so far
        // item `it`: the next id from the counter (every item, the first one too:
        // CTAs that become resident late, behind a concurrent decode kernel,
        // must not hold on to long items); decoded once here and published one
        // item ahead of its use, so no consumer and no Q copy waits on a fetch
        // at an item boundary
        auto publish = [&](int it, Item &I) -> bool {
            bool okp = true;
            int w = total;
            if (lane == 0) {
                if (it >= kItemSlots &&
                    !mbar_wait(item_empty + it % kItemSlots, (uint32_t)(((it / kItemSlots) - 1) & 1), p.wait_ns))
                    okp = false;
                else
                    w = atomicAdd(p.next_item, 1);
            }
            okp = __shfl_sync(kFull, okp ? 1 : 0, 0) != 0;
            w = __shfl_sync(kFull, w, 0);
            if (w < total) {
                I = decode_item<kB>(p, w);
            } else {
                I = Item{};
                I.live = 0;
            }
            if (lane == 0 && okp) {
                items[it % kItemSlots] = I;
                mbar_arrive(item_full + it % kItemSlots);
            }
            return okp;
        };
        // block ids of item X, 32 per chunk (lane l holds block 32*chunk + l);
        // past the sequence end (or invalid) the coordinate num_blocks is out
        // of bounds and TMA fills zeros
        auto load_ids = [&](const Item &X, int chunk) {
            const int lb = chunk * 32 + lane;
            int coord = p.num_blocks;
            if (X.live && X.valid && lb < X.nb) {
                const int32_t blk = __ldg(p.block_tables + (int64_t)X.s * p.max_blocks + lb);
                if (blk >= 0 && blk < p.num_blocks) coord = blk;
                else set_status(p.status, PA_ERR_OUT_OF_RANGE);
            }
            return coord;
        };
        Item I, I_next;
        ok = publish(0, I);
        // the first two chunks of block ids are read one item ahead, when the
        // item is published, so an item's first K copy waits on no table read
        int pre_cur = load_ids(I, 0), pre_next = load_ids(I, 1);
        for (int it = 0; ok && I.live; ++it, I = I_next) {
            if (!publish(it + 1, I_next)) { ok = false; break; }
            int ids_cur = pre_cur, ids_next = pre_next, chunk_cur = 0;
            pre_cur = load_ids(I_next, 0);
            pre_next = load_ids(I_next, 1);
            if (!I.valid) {
                if (lane == 0) set_status(p.status, PA_ERR_OUT_OF_RANGE);
                continue;
            }
            // Q: its buffer is free once every QK product of the previous item completed
            if (lane == 0) {
                if (nq >= 1 && !mbar_wait(q_empty, (uint32_t)((nq - 1) & 1), p.wait_ns)) ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(q_full, kMT * kQBytes);
                    for (int t = 0; t < kMT; ++t)
                        tma_load_4d(q_s + t * kQBytes, &tmap_q, 0, I.q0 + I.i0 + t * POS, I.g * p.group, 0, q_full);
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            ++nq;
            for (int j = 0; ok && j < I.nkv; ++j) {
                if ((j * kBlocksPerTile) / 32 != chunk_cur) {
                    ids_cur = ids_next;
                    ++chunk_cur;
                    ids_next = load_ids(I, chunk_cur + 1);
                }
                const int id0 = (j * kBlocksPerTile) & 31;
                const int cbv = __shfl_sync(kFull, ids_cur, id0 + (lane & (kBlocksPerTile - 1)));
                for (int kv = 0; kv < 2; ++kv) {
                    const int m = n + 2 * j + kv;
                    if (p.stall == PA_STALL_PRODUCER && m >= p.stall_after) {
                        stopped = true;   // test hook: entry m and later are never filled
                        ok = false;
                        break;
                    }
                    if (lane == 0 && m >= kSlots && !mbar_wait(kv_empty + slot_of(m), phase_of(m) ^ 1u, p.wait_ns))
                        ok = false;
                    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (lane == 0) mbar_arrive_expect_tx(kv_full + slot_of(m), kSlotBytes);
                    __syncwarp();
                    // lane b < kBlocksPerTile copies block b of K or V
                    if (lane < kBlocksPerTile) {
                        uint8_t *dst = kv_s + slot_of(m) * kSlotBytes + lane * kVBlockBytes;
                        if (kv)
                            tma_load_5d(dst, &tmap_v, 0, 0, 0, I.g, cbv, kv_full + slot_of(m));
                        else if (kB == 8)
                            tma_load_5d(dst, &tmap_k, 0, 0, 0, I.g, cbv, kv_full + slot_of(m));
                        else
                            tma_load_5d(dst, &tmap_k, 0, 0, I.g * kDH, 0, cbv, kv_full + slot_of(m));
                    }
                    issued_end = m + 1;
                }
            }
            n += 2 * I.nkv;
        }
        if (!ok && !stopped && lane == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            note_wait_site(p.wait_sites, PA_WAIT_PREFILL_PRODUCER);
        }
        // every copy this CTA issued has landed before the CTA may exit (these
        // waits keep the default limit whatever the test hook sets): the last Q,
        // and the last kSlots ring entries issued (earlier ones were consumed)
        if (lane == 0) {
            if (nq >= 1) mbar_wait(q_full, (uint32_t)((nq - 1) & 1));
            for (int m = issued_end > kSlots ? issued_end - kSlots : 0; m < issued_end; ++m)
                mbar_wait(kv_full + slot_of(m), phase_of(m));
        }
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer: the whole warp follows the schedule and
        // executes the MMA and commit wrappers; one elected lane issues them.  Tensor-pipe order, per KV tile j of an item:
        //   PV_0(j)  QK_0(j+1)  PV_1(j)  QK_1(j+1)
        // so the products of one M-tile run while the other tile's softmax
        // turns S into P.  QK_t(j+1) (or QK_t(0) of the next item) overwrites
        // the TMEM columns that PV_t(j) reads P_t from; the tensor pipe runs
        // one thread's MMAs in issue order, so the read precedes the overwrite.
        const uint32_t q_addr = smem_u32(q_s), kv_addr = smem_u32(kv_s);
        // descriptors: constant fields + (address >> 4) in bits 0..13
        const uint64_t dq = umma_desc_sw128(q_addr, 16, 1024);
        const uint64_t dk = umma_desc_sw128(kv_addr, 16, kKSbo);
        const uint64_t dv = umma_desc_sw128(kv_addr, kVLbo, kVSbo);
        // The K loops go out four MMAs per asm block (one 64-wide plane of the
        // swizzled operands each): fewer instructions between MMAs lets the
        // single issuing thread keep closer to the tensor pipe.
        auto issue_qk = [&](int t, int nk) {      // S_t = Q_t K^T, K in ring entry nk
            const uint32_t ko = (uint32_t)slot_of(nk) * kSlotBytes;
#pragma unroll
            for (int pl = 0; pl < D / 64; ++pl)
                umma_bf16_k64(tmem + s_col(t), dq + ((uint32_t)(t * kQBytes + pl * kPlaneQ) >> 4),
                              dk + ((ko + pl * kKPlane) >> 4), kIdescQK, pl > 0 ? 1u : 0u);
        };
        // O_t (+)= P_t V over keys 64 kq .. 64 kq + 63 (4 MMAs of 16), V in ring entry nv
        auto issue_pv = [&](int t, int nv, int kq, bool first) {
            const uint32_t vo = (uint32_t)slot_of(nv) * kSlotBytes;
            umma_bf16_tmem_a_k64(tmem + o_col(t), tmem + s_col(t) + kq * 32,
                                 dv + ((vo + kq * kVChunk) >> 4), kIdescPV, kVS1 >> 4, kVS2 >> 4,
                                 (!first || kq > 0) ? 1u : 0u);
        };
        static_assert(BN == 128, "P is released in two halves of 64 keys");
        auto commit = [&](uint64_t *bar) { umma_commit(bar); };
        bool ok = true, stopped = false;
        int n = 0, J = 0, nq = 0;
        for (int it = 0; ok; ++it) {
            Item I;
            if (!take_item(it, I)) { ok = false; break; }
            if (!I.live) break;
            if (!I.valid) continue;
            const int nkv = __shfl_sync(kFull, I.nkv, 0);
            if (p.stall == PA_STALL_CONSUMER && n >= p.stall_after) { stopped = true; ok = false; break; }
            if (!mbar_wait_warp(q_full, (uint32_t)(nq & 1), p.wait_ns) ||
                !mbar_wait_warp(kv_full + slot_of(n), phase_of(n), p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int t = 0; t < kMT; ++t) {
                issue_qk(t, n);
                commit(s_full + t);
            }
            if (nkv == 1) commit(q_empty);
            commit(kv_empty + slot_of(n));
            for (int j = 0; j < nkv; ++j) {
                const bool next = j + 1 < nkv;
                const int nv = n + 2 * j + 1, nk = n + 2 * j + 2;
                // test hook: stop, leaving ring entries unreleased, so the producer's wait runs out
                if (p.stall == PA_STALL_CONSUMER && nv >= p.stall_after) { stopped = true; ok = false; break; }
                if (!mbar_wait_warp(kv_full + slot_of(nv), phase_of(nv), p.wait_ns)) { ok = false; break; }
                for (int t = 0; t < kMT; ++t) {
                    // the item's first product into O_t overwrites it: the output
                    // warpgroup has read the previous item's O_t
                    if (j == 0 && nq > 0 && !mbar_wait_warp(o_empty + t, (uint32_t)((nq - 1) & 1), p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // the first half of P_t goes to the tensor pipe while the
                    // softmax warpgroup still computes the second
                    if (!mbar_wait_warp(p_half + t, (uint32_t)((J + j) & 1), p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(t, nv, 0, j == 0);
                    if (!mbar_wait_warp(p_full + t, (uint32_t)((J + j) & 1), p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(t, nv, 1, j == 0);
                    if (next) {
                        if (t == 0 && !mbar_wait_warp(kv_full + slot_of(nk), phase_of(nk), p.wait_ns)) { ok = false; break; }
                        tc_fence_after();
                        issue_qk(t, nk);
                        commit(s_full + t);
                    } else {
                        commit(o_full + t);
                    }
                }
                if (!ok) break;
                commit(kv_empty + slot_of(nv));
                if (next) {
                    commit(kv_empty + slot_of(nk));
                    if (j + 2 == nkv) commit(q_empty);    // the item's last QK products
                }
            }
            n += 2 * nkv;
            J += nkv;
            ++nq;
        }
        if (!ok && !stopped && lane == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            note_wait_site(p.wait_sites, PA_WAIT_PREFILL_MMA);
        }
        // drain (default limit): everything issued must finish before TMEM is released
        commit(drained);
        mbar_wait_warp(drained, 0);
        __syncwarp();
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ================= softmax warpgroup t: thread r owns row r of M-tile t
        const int t = warp >> 2;
        const int r = tid & (BM - 1);
        const int i = t * POS + (r & (POS - 1));          // position index within the CTA tile
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        bool ok = true;
        int n = 0, J = 0, no = 0;
        for (int it = 0; ok; ++it) {
            Item I;
            if (!take_item(it, I)) { ok = false; break; }
            if (!I.live) break;
            if (!I.valid) continue;
            const bool row_valid = i < I.nrows_all;
            // last visible key of this row: its position (causal) or the sequence end
            const int pos = p.causal ? I.pos_base + (row_valid ? i : I.nrows_all - 1) : I.ctx - 1;
            const int first_pos = p.causal ? I.pos_base + t * POS : I.ctx - 1;   // smallest pos of the tile
            const int t_tail = I.ctx & (kB - 1);        // valid tokens in the last block (0 = full)
            const int lb_last = (I.ctx - 1) / kB;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < I.nkv; ++j) {
                if (!mbar_wait_warp(s_full + t, (uint32_t)((J + j) & 1), p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const int key0 = j * BN;
                const bool diag = key0 + BN - 1 > first_pos;    // a key past some row of this tile
                // P = 2^(S * scale*log2e - m), bf16 pairs in registers; the first
                // tile takes its own max (key 0 is visible to every row), later
                // tiles run with the running max first: P stays <= 2^8 unless the
                // tile's max exceeds it by more than 8, and then (rarely) the row
                // moves its max, rescales O and redoes the tile from S, which is
                // intact in TMEM until P is stored over it
                // S is read whole and its max taken first, so P can go out in two
                // halves of 64 keys (the tensor pipe takes the first while the
                // second is computed); a later tile runs with the running max m:
                // P stays <= 2^8 unless the tile's max exceeds it by more than 8,
                // and then (rarely) the row moves its max and rescales O first
                uint32_t sr[BN / 32][32];
                auto mask = [&](int c) {
                    const int lim = pos - key0;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * c + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
                };
                tmem_ld32(lane_addr + s_col(t), sr[0]);
                tmem_ld32(lane_addr + s_col(t) + 32, sr[1]);
                tmem_wait_ld();
                tmem_ld32(lane_addr + s_col(t) + 64, sr[2]);
                tmem_ld32(lane_addr + s_col(t) + 96, sr[3]);
                if (diag) { mask(0); mask(1); }
                float a0 = -INFINITY, a1 = -INFINITY;
                auto max_of = [&](int c) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        a0 = fmax3(a0, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                        a1 = fmax3(a1, __uint_as_float(sr[c][e + 2]), __uint_as_float(sr[c][e + 3]));
                    }
                };
                max_of(0);
                max_of(1);
                tmem_wait_ld_regs(sr[2], sr[3]);
                if (diag) { mask(2); mask(3); }
                max_of(2);
                max_of(3);
                const float m_tile = fmaxf(a0, a1) * sl2;
                if (j == 0 && m == -INFINITY) {
                    m = m_tile == -INFINITY ? 0.f : m_tile;   // the item's first tile: its own max
                } else {
                    const bool need = m_tile > m + 8.f;
                    if (__any_sync(kFull, need)) {
                        const float m_new = need ? m_tile : m;
                        const float alpha = fast_exp2(m - m_new);
                        l *= alpha;
                        // PV_t(j-1) completed before S_t(j) was committed, so O_t is final here
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(lane_addr + o_col(t) + 32 * c, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(lane_addr + o_col(t) + 32 * c, o);
                        }
                        m = m_new;
                    }
                }
                // P = 2^(S * scale*log2e - m) for key pairs u0..u0+31 into pk; the
                // exponent's FMA and the sums as packed fp32 pairs
                const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m, -m);
                float2 ls = make_float2(0.f, 0.f);
                uint32_t pk[BN / 4];
                auto pass = [&](auto u0c) {
                    constexpr int u0 = decltype(u0c)::value;
#pragma unroll
                    for (int u = u0; u < u0 + BN / 4; ++u) {
                        const float s0 = __uint_as_float(sr[u >> 4][(2 * u) & 31]);
                        const float s1 = __uint_as_float(sr[u >> 4][(2 * u + 1) & 31]);
                        const float2 x = fma_f32x2(make_float2(s0, s1), sl2x2, negm);
                        const float p0 = fast_exp2(x.x);
                        const float p1 = fast_exp2(x.y);
                        ls = add_f32x2(ls, make_float2(p0, p1));
                        pk[u - u0] = pack_bf16x2(p0, p1);
                    }
                };
                pass(std::integral_constant<int, 0>{});
                tmem_st32(lane_addr + s_col(t), pk);
                // value rows past the context end inside the last block -> zero
                // (warpgroup 0 only; its p_half arrival orders the writes before
                // every product that reads this V tile)
                if (t == 0 && t_tail != 0) {
                    const int bb = lb_last - j * kBlocksPerTile;
                    if (bb >= 0 && bb < kBlocksPerTile) {
                        const int nv = n + 2 * j + 1;
                        if (!mbar_wait_warp(kv_full + slot_of(nv), phase_of(nv), p.wait_ns)) { ok = false; break; }
                        uint8_t *vs = kv_s + slot_of(nv) * kSlotBytes;
                        const int rows_zero = kB - t_tail;
                        const int n16 = kDH * rows_zero * 8;
                        for (int u = r; u < n16; u += BM) {
                            const int dh = u / (rows_zero * 8);
                            const int rem = u - dh * rows_zero * 8;
                            const int tok = t_tail + (rem >> 3);
                            const int off = bb * kVBlockBytes + dh * (kB * 128) + tok * 128;
                            *reinterpret_cast<uint4 *>(vs + off + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_half + t);
                // the second half of P_t over S columns 32..63
                pass(std::integral_constant<int, BN / 4>{});
                tmem_st32(lane_addr + s_col(t) + 32, pk);
                l += ls.x + ls.y;
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(p_full + t);
            }
            if (!ok) break;
            // the row's sum for the output warpgroup (double-buffered by item:
            // this buffer's previous contents, two items back, were read before
            // the output warpgroup released O_t for the item in between)
            l_s[((no & 1) * kMT + t) * BM + r] = l;
            mbar_arrive(l_full + t);
            n += 2 * I.nkv;
            J += I.nkv;
            ++no;
        }
        if (!ok && r == 0) {
            set_status(p.status, PA_ERR_TIMEOUT);
            note_wait_site(p.wait_sites, PA_WAIT_PREFILL_SOFTMAX);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    if (p.wait_at_end) grid_dependency_wait();
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

CUresult make_kv_map(CUtensorMap *map, const void *pool, int num_blocks, int kB, int hkv, int D,
                     bool all_planes) {
    auto encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_FOUND;
    // dims: d_lo(64), token(B), d_hi(D/64), head(Hkv), block; box: one block,
    // one head, one 64-column plane (B rows of 128 bytes) or all D/64 planes
    // ([plane][B rows][64] in shared memory)
    const cuuint64_t dims[5] = {64, (cuuint64_t)kB, (cuuint64_t)(D / 64), (cuuint64_t)hkv,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {(cuuint64_t)hkv * D * 2, 128, (cuuint64_t)D * 2,
                                   (cuuint64_t)kB * hkv * D * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)kB, all_planes ? (cuuint32_t)(D / 64) : 1u, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// K at B = 16 and 32, one box per cache block with every 64-column plane:
// dims d_lo(64), token within an 8-row group, 64-column quarter of a row
// (head * D/64 + plane, 128 bytes apart), 8-row group of the block, block.
// The box lands as [group][plane][8 rows][64].  (At B = 8 a block is one
// group and make_kv_map's all-planes box gives the same layout.)
CUresult make_k_map(CUtensorMap *map, const void *pool, int num_blocks, int kB, int hkv, int D) {
    auto encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[5] = {64, 8, (cuuint64_t)hkv * (D / 64), (cuuint64_t)(kB / 8), (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {(cuuint64_t)hkv * D * 2, 128, (cuuint64_t)8 * hkv * D * 2,
                                   (cuuint64_t)kB * hkv * D * 2};
    const cuuint32_t box[5] = {64, 8, (cuuint32_t)(D / 64), (cuuint32_t)(kB / 8), 1};
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

template <int D, int B>
cudaError_t launch_main(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                        const PrefillParams &prm, int grid, cudaStream_t stream) {
    const size_t smem = Shape<D>::kSmem;
    auto kern = prefill_kernel<D, B>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(grid), dim3(kThreads), smem, stream, mq, mk, mv, prm);
}

// CTA tiles a batch can produce: at least 2 * 8 positions per tile (G <= 16)
// plus one partial tile per sequence.
size_t plan_capacity(int num_seqs, int total_q) { return (size_t)total_q / 8 + num_seqs + 1; }

}  // namespace

bool prefill_tc_supported(const AttnArgs &a) {
    if (a.dtype != PA_DTYPE_BF16) return false;
    if (a.block_size != 8 && a.block_size != 16 && a.block_size != 32) return false;
    if (a.head_dim != 64 && a.head_dim != 128) return false;
    const int G = a.num_heads / a.num_kv_heads;
    if (G > 16 || log2_exact(G) < 0) return false;
    auto al = [](const void *ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; };
    return al(a.q) && al(a.out) && al(a.k_cache) && al(a.v_cache);
}

size_t prefill_workspace(int num_seqs, int total_q) {
    // [count, work counter, pad] | scratch tiles | sorted tiles
    return align_up(16 + 2 * sizeof(int2) * plan_capacity(num_seqs, total_q), 256);
}

PrefillPlanJob prefill_plan_job(const AttnArgs &a, void *workspace) {
    const int G = a.num_heads / a.num_kv_heads;
    PrefillPlanJob j;
    j.cu_seqlens_q = a.cu_seqlens_q;
    j.context_lens = a.context_lens;
    j.num_seqs = a.num_seqs;
    j.cta_shift = log2_exact(BM / G) + 1;        // kMT = 2 M-tiles per CTA tile
    j.causal = a.causal;
    j.capacity = (int)plan_capacity(a.num_seqs, a.total_q);
    j.count = static_cast<int32_t *>(workspace);
    j.next_item = j.count + 1;
    j.scratch = reinterpret_cast<int2 *>(static_cast<uint8_t *>(workspace) + 16);
    j.entries = j.scratch + j.capacity;
    return j;
}

cudaError_t launch_prefill_tc(const AttnArgs &a, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream, bool planned) {
    const int G = a.num_heads / a.num_kv_heads;
    const int pos = BM / G;
    const int pos_shift = log2_exact(pos);
    if (workspace_bytes < prefill_workspace(a.num_seqs, a.total_q)) return cudaErrorInvalidValue;
    const PrefillPlanJob job = prefill_plan_job(a, workspace);

    CUtensorMap mq, mk, mv;
    if (make_q_map(&mq, a.q, a.total_q, a.num_heads, a.head_dim, pos, G) != CUDA_SUCCESS ||
        (a.block_size == 8
             ? make_kv_map(&mk, a.k_cache, a.num_blocks, a.block_size, a.num_kv_heads, a.head_dim, true)
             : make_k_map(&mk, a.k_cache, a.num_blocks, a.block_size, a.num_kv_heads, a.head_dim)) != CUDA_SUCCESS ||
        make_kv_map(&mv, a.v_cache, a.num_blocks, a.block_size, a.num_kv_heads, a.head_dim, true) != CUDA_SUCCESS)
        return cudaErrorNotSupported;

    if (!planned) {
        cudaError_t e = cudaFuncSetAttribute(prefill_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kPrefillPlanSmem);
        if (e != cudaSuccess) return e;
        prefill_plan_kernel<<<1, kPlanThreads, kPrefillPlanSmem, stream>>>(job);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    PrefillParams prm;
    prm.cu_seqlens_q = a.cu_seqlens_q;
    prm.context_lens = a.context_lens;
    prm.block_tables = a.block_tables;
    prm.entries = job.entries;
    prm.num_entries = job.count;
    prm.next_item = job.next_item;
    prm.out = static_cast<__nv_bfloat16 *>(a.out);
    prm.num_seqs = a.num_seqs;
    prm.total_q = a.total_q;
    prm.max_q_len = a.max_q_len;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.group = G;
    prm.pos_shift = pos_shift;
    prm.max_blocks = a.max_blocks;
    prm.num_blocks = a.num_blocks;
    prm.scale_log2 = a.scale * 1.4426950408889634f;
    prm.status = a.status;
    prm.causal = a.causal;
    prm.wait_at_end = planned ? 1 : 0;
    const WaitTest &wt = wait_test();
    prm.wait_ns = wt.limit_ns;
    prm.stall = wt.stall;
    prm.stall_after = wt.after;
    prm.wait_sites = wt.sites;
    // persistent: one CTA per SM, never more CTAs than work items
    const size_t items = (size_t)job.capacity * (size_t)a.num_kv_heads;
    const int sms = device_sm_count();
    const int grid = (int)(items < (size_t)sms ? items : (size_t)sms);
    switch (a.head_dim * 100 + a.block_size) {
        case 6408: return launch_main<64, 8>(mq, mk, mv, prm, grid, stream);
        case 6416: return launch_main<64, 16>(mq, mk, mv, prm, grid, stream);
        case 6432: return launch_main<64, 32>(mq, mk, mv, prm, grid, stream);
        case 12808: return launch_main<128, 8>(mq, mk, mv, prm, grid, stream);
        case 12816: return launch_main<128, 16>(mq, mk, mv, prm, grid, stream);
        case 12832: return launch_main<128, 32>(mq, mk, mv, prm, grid, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
