// Top-K centroid selection and the cluster -> rows buckets.
//
// Step 2 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): topk over
// the centroid scores of each row.  Ties go to the lower centroid index, and
// the selected list is written sorted by (score desc, index asc).
//
// One CTA per row.  Fast path: in the pass that reads the scores, a histogram
// over the top 10 bits of their order-preserving keys (1024 buckets, each a
// half-octave of one sign); the candidates are the keys in the bucket of the
// K-th largest and above (a few dozen for Gaussian-like scores), ranked exactly
// by 64-bit (score, lower index) keys.  When that bucket is crowded (ties, odd
// distributions) the fallback is a 4-pass radix select (8 bits a pass) over
// order-preserving uint32 keys, then every key above the K-th plus the
// lowest-indexed keys equal to it.  No sort of the C scores is needed.
//
// Bucketing (masked calls): each selection (b, c) sets bit b of the cluster's
// row mask, and the first row to select a cluster appends that cluster's work
// items (chunks of `chunk` ordered positions) to the gather list.  So every
// distinct selected cluster is gathered once per call, however many rows chose
// it (step 3, the token_ordering lookup, happens in the gather kernel).
#include "internal.h"

namespace mtp {

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

constexpr int kCandCap = 512;
// Fast-path buckets: the top 10 bits of the order-preserving key (sign, exponent
// and one mantissa bit: half-octaves).
constexpr int kKeyBits = 10;
constexpr int kKeyBuckets = 1 << kKeyBits;
constexpr int kKeyShift = 32 - kKeyBits;
static_assert(kKeyBuckets % kTopkThreads == 0, "whole buckets per thread");
static_assert(kCandCap * 8 <= kKeyBuckets * 4, "the candidates reuse the histogram's memory");

__device__ __forceinline__ unsigned long long select_key(uint32_t ord, int c)
{
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)c);
}

// Bucketing of row b's K selections `sel` (shared memory; see the file comment), one
// warp per 32 selections: each lane sets its row-mask bit and counts the cluster's
// rows; the first selectors of their clusters then reserve their work items with one
// atomicAdd per warp on the item count (a warp-wide prefix sum of their item counts),
// not one per cluster on the same word.
__device__ __forceinline__ void bucket_selections(const TopkParams &p, int b, const int32_t *sel)
{
    const int lane = threadIdx.x & (kWarp - 1), warp = threadIdx.x / kWarp;
    for (int i0 = warp * kWarp; i0 < p.K; i0 += kTopkThreads) {
        const int c = i0 + lane < p.K ? sel[i0 + lane] : -1;
        int n = 0;
        if (c >= p.c_begin && c < p.c_end) {   // else another shard's cluster (or no lane)
            atomicOr(&p.rowmask[(size_t)c * p.W + (b >> 5)], 1u << (b & 31));
            int lo, hi;
            if (atomicAdd(&p.ccount[c], 1) == 0 &&
                cluster_range(p.offsets, p.V, p.S, c, &lo, &hi, p.ctrl + kCtrlError) && hi > lo)
                n = (hi - lo + p.chunk - 1) / p.chunk;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
        if (total == 0) continue;
        uint32_t base = 0;
        if (lane == kWarp - 1) base = atomicAdd(p.ctrl + kCtrlItems, (uint32_t)total);
        base = __shfl_sync(0xffffffffu, base, kWarp - 1) + (uint32_t)(incl - n);
        if (n == 0) continue;
        // Ascending offsets cannot overflow the list (it is sized for V / chunk + C items);
        // overlapping ranges can, so a cluster that does not fit is reported and dropped.
        if (base + (uint32_t)n > (uint32_t)p.items_cap) {
            atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_OFFSETS);
        } else {
            for (int j = 0; j < n; ++j) p.items[base + j] = make_int2(c, j * p.chunk);
        }
    }
}

__global__ void __launch_bounds__(kTopkThreads) k_topk(TopkParams p)
{
    extern __shared__ uint32_t sm[];
    uint32_t *keys = sm;                                      // [C]
    int32_t *sel = reinterpret_cast<int32_t *>(sm + p.C);     // [K]
    // the histogram, then (once scanned) the candidate keys in the same memory
    __shared__ __align__(8) uint32_t hist[kKeyBuckets];
    unsigned long long *s_cand = reinterpret_cast<unsigned long long *>(hist);
    __shared__ int s_scan[kWarp + 1];
    __shared__ uint32_t s_digit, s_above;

    const int b = blockIdx.x, tid = threadIdx.x;
    for (int i = tid; i < kKeyBuckets; i += kTopkThreads) hist[i] = 0u;
    __syncthreads();
    // the first selector of a cluster reads its range from the offsets table
    if (p.rowmask) prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    // the scores are written by the projection kernel that precedes this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const float *row = p.scores + (size_t)b * p.C;

    // Fast path: one pass reads the scores, keeps their order-preserving keys and
    // histograms them by the keys' top bits (sign, exponent and one mantissa bit:
    // buckets a half-octave wide, monotone in the score); the candidates are the
    // keys in the bucket of the K-th largest and above, ranked exactly by 64-bit
    // (score, lower index) keys.
    for (int c = tid; c < p.C; c += kTopkThreads) {
        const float v = p.bf16_scores ? round_bf16(row[c]) : row[c];
        const uint32_t k = ord_key(v);
        keys[c] = k;
        atomicAdd(&hist[k >> kKeyShift], 1u);
    }
    __syncthreads();
    // thread t owns the per buckets below kKeyBuckets - per*t, largest first
    {
        constexpr int per = kKeyBuckets / kTopkThreads;
        uint32_t loc[per], sum = 0u;
#pragma unroll
        for (int j = 0; j < per; ++j) {
            loc[j] = hist[kKeyBuckets - 1 - (tid * per + j)];
            sum += loc[j];
        }
        int total;
        const uint32_t excl = (uint32_t)cta_exclusive_scan((int)sum, s_scan, &total);
        const uint32_t need = (uint32_t)p.K;
        if (excl < need && need <= excl + sum) {
            uint32_t run = excl;
#pragma unroll
            for (int j = 0; j < per; ++j) {
                if (run + loc[j] >= need) {
                    s_digit = (uint32_t)(kKeyBuckets - 1 - (tid * per + j));
                    s_above = run + loc[j];   // candidates: this bucket and every one above
                    break;
                }
                run += loc[j];
            }
        }
    }
    __syncthreads();
    const uint32_t kbucket = s_digit;
    const int ncand = (int)s_above;
    if (ncand <= kCandCap) {
        // compaction without atomics: each warp counts its hits over its columns (ballots),
        // one prefix over the warps gives each warp its first slot, and a second pass
        // writes the candidates (their order does not matter to the ranking)
        const int lane = tid & (kWarp - 1), warp = tid / kWarp;
        int whits = 0;
        for (int c0 = 0; c0 < p.C; c0 += kTopkThreads) {
            const int c = c0 + tid;
            const bool hit = c < p.C && (keys[c] >> kKeyShift) >= kbucket;
            whits += __popc(__ballot_sync(0xffffffffu, hit));
        }
        if (lane == 0) s_scan[warp] = whits;
        __syncthreads();
        int slot = 0;
        for (int w = 0; w < warp; ++w) slot += s_scan[w];
        for (int c0 = 0; c0 < p.C; c0 += kTopkThreads) {
            const int c = c0 + tid;
            const uint32_t k = c < p.C ? keys[c] : 0u;
            const bool hit = c < p.C && (k >> kKeyShift) >= kbucket;
            const unsigned bal = __ballot_sync(0xffffffffu, hit);
            if (hit) s_cand[slot + __popc(bal & ((1u << lane) - 1u))] = select_key(k, c);
            slot += __popc(bal);
        }
        __syncthreads();
        // rank of each candidate = candidates with a larger key; with few candidates four
        // threads (an aligned group of lanes) split one candidate's comparisons.  The
        // thread that finds a rank below K stores and buckets that selection at once.
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
            if (q == 0 && rank < p.K) {
                const int c = (int)(0xffffffffu - (uint32_t)(ki & 0xffffffffull));
                p.topk[(size_t)b * p.K + rank] = c;
                sel[rank] = c;
            }
        }
        if (p.rowmask == nullptr) return;
        __syncthreads();
        bucket_selections(p, b, sel);
        return;
    }

    // Radix select: after the passes, `prefix` is the K-th largest key and
    // `need` the number of keys equal to it that belong to the selection.
    uint32_t prefix = 0u, mask = 0u, need = (uint32_t)p.K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads)
            hist[i] = 0u;
        __syncthreads();
        // Scores crowd into few bins of the high digits, so lanes that hit the same
        // bin combine their increments (one shared atomic per bin per warp).
        for (int c0 = 0; c0 < p.C; c0 += kTopkThreads) {
            const int c = c0 + tid;
            const uint32_t u = c < p.C ? keys[c] : 0u;
            const bool hit = c < p.C && (u & mask) == prefix;
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
                        s_digit = 255u - (uint32_t)(lane * 8 + j);
                        s_above = run;
                        break;
                    }
                    run += loc[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 0xffu << shift;
        need -= s_above;
    }
    const uint32_t kth = prefix;

    // Selection in index order: thread t owns a contiguous index range, so an
    // exclusive scan over threads orders both the equal keys (lowest index
    // first) and the output positions.
    const int per = (p.C + kTopkThreads - 1) / kTopkThreads;
    const int c_beg = min(p.C, tid * per), c_end = min(p.C, c_beg + per);
    int n_gt = 0, n_eq = 0;
    for (int c = c_beg; c < c_end; ++c) {
        const uint32_t u = keys[c];
        n_gt += u > kth;
        n_eq += u == kth;
    }
    int total;
    const int eq_before = cta_exclusive_scan(n_eq, s_scan, &total);
    const int take_eq = max(0, min(n_eq, (int)need - eq_before));
    int pos = cta_exclusive_scan(n_gt + take_eq, s_scan, &total);
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
    for (int i = tid; i < p.K; i += kTopkThreads) {
        const int ci = sel[i];
        const uint32_t ki = keys[ci];
        int rank = 0;
        for (int j = 0; j < p.K; ++j) {
            const int cj = sel[j];
            const uint32_t kj = keys[cj];
            rank += (kj > ki) || (kj == ki && cj < ci);
        }
        p.topk[(size_t)b * p.K + rank] = ci;
    }

    if (p.rowmask == nullptr)
        return;
    bucket_selections(p, b, sel);
}

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s)
{
    const size_t smem = (size_t)(p.C + p.K) * sizeof(uint32_t);
    cudaError_t e = allow_smem((const void *)k_topk, smem);
    if (e != cudaSuccess)
        return e;
    return launch_dependent(k_topk, dim3(p.B), dim3(kTopkThreads), smem, s, p);
}

}  // namespace mtp
