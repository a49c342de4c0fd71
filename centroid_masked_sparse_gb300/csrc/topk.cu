// Top-K centroid selection and the cluster -> rows buckets.
//
// Step 2 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): topk over
// the centroid scores of each row.  Ties go to the lower centroid index, and
// the selected list is written sorted by (score desc, index asc).
//
// One CTA per row; the exact selection itself (a histogram over the keys' top
// bits, then a ranking of the few candidates, with a radix-select fallback) is
// select_topk_row in topk_select.cuh.
//
// Bucketing (masked calls): each selection (b, c) sets bit b of the cluster's
// row mask, and the first row to select a cluster appends that cluster's work
// items (chunks of `chunk` ordered positions) to the gather list.  So every
// distinct selected cluster is gathered once per call, however many rows chose
// it (step 3, the token_ordering lookup, happens in the gather kernel).
#include "topk_select.cuh"

namespace mtp {

// Bucketing of row b's K selections `sel` (shared memory; see the file comment), one
// selection a thread: each sets its row-mask bit and counts the cluster's rows; the
// first selectors of their clusters then reserve their work items with one atomicAdd
// per CTA on the item count (a CTA-wide prefix sum of their item counts).  All rows
// reach this point at about the same time, and atomics on one word serialise: one per
// warp measured several microseconds slower than one per CTA with K = 128, B = 256.
__device__ __forceinline__ void bucket_selections(const TopkParams &p, int b, const int32_t *sel, TopkShared &ts)
{
    for (int i0 = 0; i0 < p.K; i0 += kTopkThreads) {
        const int i = i0 + (int)threadIdx.x;
        const int c = i < p.K ? sel[i] : -1;
        int n = 0;
        if (c >= p.c_begin && c < p.c_end) {   // else another shard's cluster (or no selection)
            atomicOr(&p.rowmask[(size_t)c * p.W + (b >> 5)], 1u << (b & 31));
            int lo, hi;
            if (atomicAdd(&p.ccount[c], 1) == 0 &&
                cluster_range(p.offsets, p.V, p.S, c, &lo, &hi, p.ctrl + kCtrlError) && hi > lo)
                n = (hi - lo + p.chunk - 1) / p.chunk;
        }
        int total;
        const int excl = cta_exclusive_scan(n, ts.scan, &total);
        if (total == 0) continue;   // uniform over the CTA
        if (threadIdx.x == 0) ts.above = atomicAdd(p.ctrl + kCtrlItems, (uint32_t)total);
        __syncthreads();
        const uint32_t base = ts.above + (uint32_t)excl;
        __syncthreads();   // every thread has read the base before the next round sets it
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
    __shared__ TopkShared ts;

    const int b = blockIdx.x;
    topk_clear(ts);
    // the first selector of a cluster reads its range from the offsets table
    if (p.rowmask) prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    // the scores are written by the projection kernel that precedes this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    select_topk_row(p.scores + (size_t)b * p.C, p.C, p.K, p.bf16_scores != 0, keys, sel, p.topk + (size_t)b * p.K,
                    ts);
    if (p.rowmask == nullptr) return;
    bucket_selections(p, b, sel, ts);
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
