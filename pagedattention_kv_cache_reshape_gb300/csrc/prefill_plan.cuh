// prefill_plan.cuh -- the work list of the tcgen05 prefill kernel, built by one
// CTA of any size.  Used by the prefill kernel's own plan launch and, for a
// batch with decode rows too, by one extra CTA of the decode plan kernel, so
// a mixed batch needs a single plan launch.
//
// A work item is a CTA tile: 2 M-tiles of 128 rows, i.e. 2 * (128 / G)
// consecutive query positions of one sequence with q_len >= 2, for one
// kv-head.  The tiles are listed in sequence order, then counting-sorted on
// their number of 128-key tiles, most first, so the persistent CTAs take the
// longest work first and finish together.
#pragma once

#include <stdint.h>

namespace pa {

constexpr int kPrefillKeysPerTile = 128;      // keys per KV tile of the prefill kernel
constexpr int kPrefillCostBuckets = 1024;
constexpr int kPrefillPlanSmemTiles = 4096;   // tiles staged in shared memory (else in `scratch`)
// shared memory of prefill_plan_block: warp totals | buckets | tiles | costs
constexpr int kPrefillPlanSmem = 32 * 4 + kPrefillCostBuckets * 4 + kPrefillPlanSmemTiles * 8 +
                                 kPrefillPlanSmemTiles * 2;

struct PrefillPlanJob {
    const int32_t *cu_seqlens_q;
    const int32_t *context_lens;
    int num_seqs;
    int cta_shift;        // log2(query positions per CTA tile)
    int causal;
    int capacity;         // tiles `scratch` and `entries` hold
    int2 *scratch;
    int2 *entries;        // (sequence, CTA tile), most KV tiles first
    int32_t *count;
    int32_t *next_item;   // the persistent kernel's work counter, reset here
};

// KV tiles a CTA tile needs: keys up to its last row's position (causal) or
// the whole sequence; 0 marks a tile the main kernel rejects.
__device__ __forceinline__ int prefill_tile_kv_tiles(int q_len, int ctx, int tile, int cta_shift,
                                                     int causal) {
    const int i0 = tile << cta_shift;
    const int nrows = min(1 << cta_shift, q_len - i0);
    if (ctx <= 0 || q_len < 2 || q_len > ctx || nrows <= 0) return 0;
    const int pos_last = causal ? ctx - q_len + i0 + nrows - 1 : ctx - 1;
    return pos_last / kPrefillKeysPerTile + 1;
}

// The whole plan, by the calling CTA (blockDim.x a multiple of 32, at most
// 1024, and a divisor of kPrefillCostBuckets); `smem` holds kPrefillPlanSmem
// bytes, 8-byte aligned.
__device__ inline void prefill_plan_block(const PrefillPlanJob &j, uint8_t *smem) {
    int *warp_tot = reinterpret_cast<int *>(smem);
    int *bucket = warp_tot + 32;
    int2 *tiles_s = reinterpret_cast<int2 *>(bucket + kPrefillCostBuckets);
    uint16_t *cost_s = reinterpret_cast<uint16_t *>(tiles_s + kPrefillPlanSmemTiles);
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = nthr >> 5;
    const bool in_smem = j.capacity <= kPrefillPlanSmemTiles;
    int2 *tiles = in_smem ? tiles_s : j.scratch;
    const int pos = 1 << j.cta_shift;
    auto bucket_of_cost = [](int c) {
        // bucket b holds the tiles with kPrefillCostBuckets-1-b KV tiles (the last
        // bucket collects everything longer): ascending buckets = most work first
        return kPrefillCostBuckets - 1 - min(c, kPrefillCostBuckets - 1);
    };
    for (int b = tid; b < kPrefillCostBuckets; b += nthr) bucket[b] = 0;
    __syncthreads();
    int running = 0;
    for (int base = 0; base < j.num_seqs; base += nthr) {
        const int s = base + tid;
        int nt = 0, q_len = 0, ctx = 0;
        if (s < j.num_seqs) {
            q_len = __ldg(j.cu_seqlens_q + s + 1) - __ldg(j.cu_seqlens_q + s);
            ctx = __ldg(j.context_lens + s);
            if (q_len > 1) nt = (q_len + pos - 1) >> j.cta_shift;
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
        for (int w = 0; w < nwarps; ++w) {
            if (w < warp) warp_off += warp_tot[w];
            chunk_tot += warp_tot[w];
        }
        const int first = running + warp_off + incl - nt;
        for (int t = 0; t < nt; ++t) {
            if (first + t >= j.capacity) break;
            const int b = bucket_of_cost(prefill_tile_kv_tiles(q_len, ctx, t, j.cta_shift, j.causal));
            tiles[first + t] = make_int2(s, t);
            if (in_smem) cost_s[first + t] = (uint16_t)b;
            atomicAdd(&bucket[b], 1);
        }
        running += chunk_tot;
        __syncthreads();
    }
    const int total = running < j.capacity ? running : j.capacity;
    // exclusive scan of the buckets, kPrefillCostBuckets / nthr per thread
    const int per = kPrefillCostBuckets / nthr;
    int sum = 0;
    for (int k = 0; k < per; ++k) sum += bucket[tid * per + k];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int off = incl - sum;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    __syncthreads();   // every thread has read its buckets before they are rewritten
    for (int k = 0; k < per; ++k) {
        const int c = bucket[tid * per + k];
        bucket[tid * per + k] = off;
        off += c;
    }
    __syncthreads();
    for (int e = tid; e < total; e += nthr) {
        const int2 v = tiles[e];
        int b;
        if (in_smem) {
            b = cost_s[e];
        } else {
            const int q0 = __ldg(j.cu_seqlens_q + v.x);
            b = bucket_of_cost(prefill_tile_kv_tiles(__ldg(j.cu_seqlens_q + v.x + 1) - q0,
                                                     __ldg(j.context_lens + v.x), v.y, j.cta_shift,
                                                     j.causal));
        }
        j.entries[atomicAdd(&bucket[b], 1)] = v;
    }
    if (tid == 0) {
        *j.count = total;
        *j.next_item = 0;
    }
}

}  // namespace pa
