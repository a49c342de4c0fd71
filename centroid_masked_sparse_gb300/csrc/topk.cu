// Top-K centroid selection and the cluster -> rows buckets.
//
// Step 2 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): topk over
// the centroid scores of each row.  Ties go to the lower centroid index, and
// the selected list is written sorted by (score desc, index asc).
//
// One CTA per row.  The K-th largest score is found by a 4-pass radix select
// (8 bits a pass) over order-preserving uint32 keys held in shared memory; the
// selection is then every key above it plus the lowest-indexed keys equal to
// it.  No sort of the C scores is needed.
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

__global__ void __launch_bounds__(kTopkThreads) k_topk(TopkParams p)
{
    extern __shared__ uint32_t sm[];
    uint32_t *keys = sm;                                      // [C]
    int32_t *sel = reinterpret_cast<int32_t *>(sm + p.C);     // [K]
    __shared__ uint32_t hist[256];
    __shared__ int s_scan[kWarp + 1];
    __shared__ uint32_t s_digit, s_above;

    const int b = blockIdx.x, tid = threadIdx.x;
    const float *row = p.scores + (size_t)b * p.C;
    for (int c = tid; c < p.C; c += kTopkThreads)
        keys[c] = ord_key(row[c]);

    // Radix select: after the passes, `prefix` is the K-th largest key and
    // `need` the number of keys equal to it that belong to the selection.
    uint32_t prefix = 0u, mask = 0u, need = (uint32_t)p.K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kTopkThreads)
            hist[i] = 0u;
        __syncthreads();
        for (int c = tid; c < p.C; c += kTopkThreads) {
            const uint32_t u = keys[c];
            if ((u & mask) == prefix)
                atomicAdd(&hist[(u >> shift) & 255u], 1u);
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
    for (int i = tid; i < p.K; i += kTopkThreads) {
        const int c = sel[i];
        atomicOr(&p.rowmask[(size_t)c * p.W + (b >> 5)], 1u << (b & 31));
        if (atomicAdd(&p.ccount[c], 1) == 0) {
            int lo, hi;
            if (cluster_range(p.offsets, p.V, p.S, c, &lo, &hi, p.ctrl + kCtrlError) && hi > lo) {
                const int n = (hi - lo + p.chunk - 1) / p.chunk;
                const uint32_t base = atomicAdd(p.ctrl + kCtrlItems, (uint32_t)n);
                // Ascending offsets cannot overflow the list (it is sized for V / chunk + C
                // items); overlapping ranges can, so they are reported and dropped.
                if (base + (uint32_t)n > (uint32_t)p.items_cap) {
                    atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_OFFSETS);
                } else {
                    for (int j = 0; j < n; ++j)
                        p.items[base + j] = make_int2(c, j * p.chunk);
                }
            }
        }
    }
}

cudaError_t launch_topk(const TopkParams &p, cudaStream_t s)
{
    const size_t smem = (size_t)(p.C + p.K) * sizeof(uint32_t);
    cudaError_t e = allow_smem((const void *)k_topk, smem);
    if (e != cudaSuccess)
        return e;
    k_topk<<<p.B, kTopkThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mtp
