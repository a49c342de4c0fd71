// Exact top-K selection of one row of centroid scores by one CTA of
// kTopkThreads threads: the K largest scores, ties to the lower centroid index.
// Used by the top-K kernel (one CTA per row) and by the fused small-batch
// kernel (every CTA selects the row it gathers for).
//
// Step 2 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): topk over
// the centroid scores of each row.
//
// Fast path: in the pass that reads the scores, a histogram over the top 10 bits
// of their order-preserving keys (1024 buckets, each a half-octave of one sign);
// the candidates are the keys in the bucket of the K-th largest and above (a few
// dozen for Gaussian-like scores), ranked exactly by 64-bit (score, lower index)
// keys.  When that bucket is crowded (ties, odd distributions) the fallback is a
// 4-pass radix select (8 bits a pass) over the order-preserving uint32 keys, then
// every key above the K-th plus the lowest-indexed keys equal to it.  No sort of
// the C scores is needed.
#pragma once

#include "internal.h"

namespace mtp {

constexpr int kCandCap = 512;
// Fast-path buckets: the top 10 bits of the order-preserving key (sign, exponent
// and one mantissa bit: half-octaves).
constexpr int kKeyBits = 10;
constexpr int kKeyBuckets = 1 << kKeyBits;
constexpr int kKeyShift = 32 - kKeyBits;
static_assert(kKeyBuckets == 4 * kTopkThreads, "the bucket search reads four buckets a thread");
static_assert(kCandCap * 8 <= kKeyBuckets * 4, "the candidates reuse the histogram's memory");

// Static shared memory of one selection.
struct TopkShared {
    // the histogram, then (once scanned) the candidate keys in the same memory
    __align__(16) uint32_t hist[kKeyBuckets];
    uint32_t wsum[kTopkThreads / kWarp];   // the bucket search's per-warp counts
    int scan[kWarp + 1];
    uint32_t digit, above;
};

// Exclusive prefix sum over the CTA (kTopkThreads threads); *total gets the sum.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *s_scan, int *total)
{
    constexpr int NW = kTopkThreads / kWarp;
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    int x = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == kWarp - 1) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < NW ? s_scan[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < NW) s_scan[lane] = wi - w;
        if (lane == NW - 1) s_scan[kWarp] = wi;
    }
    __syncthreads();
    const int excl = s_scan[warp] + x - v;
    *total = s_scan[kWarp];
    __syncthreads();
    return excl;
}

__device__ __forceinline__ unsigned long long select_key(uint32_t ord, int c)
{
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)c);
}

// Clears the histogram of a selection; call it (every thread of the CTA) before
// select_topk_row, e.g. while the kernel still waits for the scores.
__device__ __forceinline__ void topk_clear(TopkShared &ts)
{
    for (int i = threadIdx.x; i < kKeyBuckets; i += kTopkThreads) ts.hist[i] = 0u;
}

// Rows of at most this many scores take an instantiation whose loops over the
// row have fixed trip counts (fully unrolled: measured ~15 % faster at C = 2048).
constexpr int kTopkSmallC = 8 * kTopkThreads;

template <bool SMALL>
__device__ __forceinline__ void select_topk_row_impl(const float *row, int C, int K, bool bf16_scores,
                                                     uint32_t *keys, int32_t *sel, int32_t *sorted_out,
                                                     TopkShared &ts)
{
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid / kWarp;
    uint32_t *hist = ts.hist;
    unsigned long long *s_cand = reinterpret_cast<unsigned long long *>(ts.hist);
    if (tid == 0) ts.above = 0u;   // the candidate count of the compaction below
    __syncthreads();               // the histogram's clearing is visible

    // one pass reads the scores (eight loads in flight per thread before any is used),
    // keeps their order-preserving keys and histograms them by the keys' top bits
    // (buckets a half-octave wide, monotone in the score)
    constexpr int kLoads = 8;
    const int c_lim = SMALL ? kTopkSmallC : C;
    for (int c0 = 0; c0 < c_lim; c0 += kLoads * kTopkThreads) {
        float v[kLoads];
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
            const int c = c0 + j * kTopkThreads + tid;
            v[j] = c < C ? __ldcg(row + c) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
            const int c = c0 + j * kTopkThreads + tid;
            if (c < C) {
                const uint32_t k = ord_key(bf16_scores ? round_bf16(v[j]) : v[j]);
                keys[c] = k;
                atomicAdd(&hist[k >> kKeyShift], 1u);
            }
        }
    }
    __syncthreads();
    // the bucket of the K-th largest key, found by the whole CTA: thread t holds buckets
    // 1023-4t down to 1020-4t (one 16-byte load), a scan over the lanes and one over the
    // warps' totals give the count of keys above each thread's buckets, and the thread
    // whose buckets reach the K-th key finds the bucket among its four.  (One warp summing
    // 32 buckets a lane took ~3000 cycles on GB300, this ~500.)
    {
        const uint4 q = reinterpret_cast<const uint4 *>(hist)[kKeyBuckets / 4 - 1 - tid];
        const uint32_t sum = q.x + q.y + q.z + q.w;
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == kWarp - 1) ts.wsum[warp] = incl;
        __syncthreads();
        uint32_t above = incl - sum;
#pragma unroll
        for (int w = 0; w < kTopkThreads / kWarp; ++w) above += w < warp ? ts.wsum[w] : 0u;
        const uint32_t need = (uint32_t)K;
        if (above < need && above + sum >= need) {
            const int b0 = kKeyBuckets - 1 - 4 * tid;
            uint32_t run = above, d = (uint32_t)(b0 - 3);
            if ((run += q.w) >= need) d = (uint32_t)b0;
            else if ((run += q.z) >= need) d = (uint32_t)(b0 - 1);
            else if ((run += q.y) >= need) d = (uint32_t)(b0 - 2);
            else run += q.x;
            ts.digit = d;
            ts.scan[kWarp] = (int)run;   // candidates: this bucket and every one above
        }
    }
    __syncthreads();
    const uint32_t kbucket = ts.digit;
    const int ncand = ts.scan[kWarp];
    if (ncand <= kCandCap) {
        // compaction: each warp counts its hits (ballots over its columns), takes that many
        // consecutive slots with one shared atomic, and writes them in a second pass (the
        // slots' order does not matter to the ranking)
        int whits = 0;
#pragma unroll(SMALL ? 8 : 1)
        for (int c0 = 0; c0 < c_lim; c0 += kTopkThreads) {
            const int c = c0 + tid;
            whits += __popc(__ballot_sync(0xffffffffu, c < C && (keys[c] >> kKeyShift) >= kbucket));
        }
        uint32_t slot = 0u;
        if (lane == 0 && whits) slot = atomicAdd(&ts.above, (uint32_t)whits);
        slot = __shfl_sync(0xffffffffu, slot, 0);
#pragma unroll(SMALL ? 8 : 1)
        for (int c0 = 0; c0 < c_lim && whits; c0 += kTopkThreads) {
            const int c = c0 + tid;
            const uint32_t k = c < C ? keys[c] : 0u;
            const bool hit = c < C && (k >> kKeyShift) >= kbucket;
            const unsigned bal = __ballot_sync(0xffffffffu, hit);
            if (hit) s_cand[slot + __popc(bal & ((1u << lane) - 1u))] = select_key(k, c);
            slot += __popc(bal);
        }
        __syncthreads();
        // rank of each candidate = candidates with a larger key; with few candidates four
        // threads (an aligned group of lanes) split one candidate's comparisons
        const int tpc = ncand <= kTopkThreads / 4 ? 4 : 1;
        const int q = tid % tpc;
        for (int i = tid / tpc; i < ncand; i += kTopkThreads / tpc) {
            const unsigned long long ki = s_cand[i];
            int rank = 0;
#pragma unroll 4
            for (int j = q; j < ncand; j += tpc) rank += s_cand[j] > ki;
            if (tpc == 4) {
                const unsigned grp = 0xfu << ((tid & (kWarp - 1)) & ~3);
                rank += __shfl_xor_sync(grp, rank, 1);
                rank += __shfl_xor_sync(grp, rank, 2);
            }
            if (q == 0 && rank < K) {
                const int c = (int)(0xffffffffu - (uint32_t)(ki & 0xffffffffull));
                if (sorted_out) sorted_out[rank] = c;
                sel[rank] = c;
            }
        }
        __syncthreads();
        return;
    }

    // Radix select: after the passes, `prefix` is the K-th largest key and
    // `need` the number of keys equal to it that belong to the selection.
    uint32_t prefix = 0u, mask = 0u, need = (uint32_t)K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads)
            hist[i] = 0u;
        __syncthreads();
        // Scores crowd into few bins of the high digits, so lanes that hit the same
        // bin combine their increments (one shared atomic per bin per warp).
        for (int c0 = 0; c0 < C; c0 += kTopkThreads) {
            const int c = c0 + tid;
            const uint32_t u = c < C ? keys[c] : 0u;
            const bool hit = c < C && (u & mask) == prefix;
            const uint32_t bin = (u >> shift) & 255u;
            const unsigned peers = __match_any_sync(0xffffffffu, hit ? bin : 256u + (tid & 31));
            if (hit && (tid & 31) == __ffs(peers) - 1)
                atomicAdd(&hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (tid < kWarp) {
            // lane l scans bins 255-8l .. 248-8l (largest digits first)
            const int lane = tid;
            uint32_t loc[8], sum = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                loc[j] = hist[255 - (lane * 8 + j)];
                sum += loc[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - sum;
            if (excl < need && need <= incl) {
                uint32_t run = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + loc[j] >= need) {
                        ts.digit = 255u - (uint32_t)(lane * 8 + j);
                        ts.above = run;
                        break;
                    }
                    run += loc[j];
                }
            }
        }
        __syncthreads();
        prefix |= ts.digit << shift;
        mask |= 0xffu << shift;
        need -= ts.above;
    }
    const uint32_t kth = prefix;

    // Selection in index order: thread t owns a contiguous index range, so an
    // exclusive scan over threads orders both the equal keys (lowest index
    // first) and the output positions.
    const int per = (C + kTopkThreads - 1) / kTopkThreads;
    const int c_beg = min(C, tid * per), c_end = min(C, c_beg + per);
    int n_gt = 0, n_eq = 0;
    for (int c = c_beg; c < c_end; ++c) {
        const uint32_t u = keys[c];
        n_gt += u > kth;
        n_eq += u == kth;
    }
    int total;
    const int eq_before = cta_exclusive_scan(n_eq, ts.scan, &total);
    const int take_eq = max(0, min(n_eq, (int)need - eq_before));
    int pos = cta_exclusive_scan(n_gt + take_eq, ts.scan, &total);
    int eq_seen = 0;
    for (int c = c_beg; c < c_end; ++c) {
        const uint32_t u = keys[c];
        bool take = u > kth;
        if (u == kth) {
            take = eq_seen < take_eq;
            ++eq_seen;
        }
        if (take)
            sel[pos++] = c;
    }
    __syncthreads();

    // Sorted output: the rank of each selected centroid under (key desc, index asc).
    if (sorted_out) {
        for (int i = tid; i < K; i += kTopkThreads) {
            const int ci = sel[i];
            const uint32_t ki = keys[ci];
            int rank = 0;
            for (int j = 0; j < K; ++j) {
                const int cj = sel[j];
                const uint32_t kj = keys[cj];
                rank += (kj > ki) || (kj == ki && cj < ci);
            }
            sorted_out[rank] = ci;
        }
    }
    __syncthreads();
}

// Selects the K largest of row[0..C) (rounded to bf16 first with bf16_scores).
// On return (after a final __syncthreads) sel[0..K) holds the selected centroids,
// in a deterministic order (by rank on the fast path, by index on the fallback),
// and, when sorted_out is not null, sorted_out[0..K) holds them sorted by (score
// desc, index asc).  keys: shared [C]; sel: shared [K].  The histogram must have
// been cleared by topk_clear.  Every thread of the CTA must call it.
__device__ __forceinline__ void select_topk_row(const float *row, int C, int K, bool bf16_scores, uint32_t *keys,
                                                int32_t *sel, int32_t *sorted_out, TopkShared &ts)
{
    if (C <= kTopkSmallC)
        select_topk_row_impl<true>(row, C, K, bf16_scores, keys, sel, sorted_out, ts);
    else
        select_topk_row_impl<false>(row, C, K, bf16_scores, keys, sel, sorted_out, ts);
}

}  // namespace mtp
