// Fused top-K, candidate gather and sparse dot products for small batches.
//
// Steps 2-4 and the finishes of Gemma4MTPMaskedEmbedder._select_and_score /
// get_top_tokens / forward ("Add Gemma4 MTP speculative decoding with centroids
// masking", vLLM gemma4_mtp.py), in one kernel that runs behind the projection.
//
// With a few rows the call is a chain of dependent latencies, not a stream of
// bytes: at one row it moves 19 MB, under 3 us of HBM time.  So this kernel
// drops the separate top-K kernel, its bucketing atomics and the work-item list.
// Every CTA serves one row (CTA j -> row j mod B, so a row's CTAs spread over
// the SMs): it reads that row's C scores from L2 and selects the row's top-K
// itself (the same exact selection as the top-K kernel, so every CTA of a row
// finds the same set), numbers the row's candidates (its selected clusters'
// ordered positions, cluster after cluster) and takes an equal slice of them.
// Each warp then takes a contiguous part of the slice: its lanes look up 32
// token ids at once, and it streams the candidates' embedding rows straight into
// registers (16-byte loads; two batches of 1 to 8 rows in flight, more for
// shorter rows) and dots each with the hidden row held in shared memory.  The argmax finish folds (logit, lower id) keys per
// warp, per CTA (shared 64-bit atomicMax) and per row (one global atomicMax),
// and the last CTA to finish (a ticket, no wait) turns the keys into token ids;
// the scatter finish stores each logit into the -inf-filled row.
//
// Rows that selected the same cluster each read it: at these batch sizes two
// rows rarely share a cluster (at B = 8 and K = 32 of 2048, 5 % of the pairs).
#include <algorithm>

#include "topk_select.cuh"

namespace mtp {

namespace {

template <int NCH>
__device__ __forceinline__ void load_row(uint4 (&e)[NCH], const uint16_t *row, int hv, int lane)
{
#pragma unroll
    for (int q = 0; q < NCH; ++q) {
        const int idx = q * kWarp + lane;
        e[q] = idx < hv ? ld_stream16(row + (size_t)idx * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <int NCH>
__device__ __forceinline__ float dot_row(const uint4 (&e)[NCH], const uint4 *hs, int hv, int lane)
{
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < NCH; ++q) {
        const int idx = q * kWarp + lane;
        if (idx < hv) acc = dot8_bf16_mixed(e[q], hs[idx], acc);
    }
    return warp_sum(acc);
}

// Candidates a warp loads together: 16-byte pieces per lane per row NCH, rows R.
__host__ __device__ constexpr int select_gather_batch(int nch)
{
    return nch <= 1 ? 8 : nch == 2 ? 4 : nch <= 4 ? 2 : 1;
}
static_assert(kWarp % select_gather_batch(1) == 0, "a batch never straddles a refill of the lanes' ids");

template <int NCH, bool SCATTER>
__global__ void __launch_bounds__(kTopkThreads) k_select_gather(const GatherParams p)
{
    extern __shared__ uint4 dyn[];
    __shared__ TopkShared ts;
    __shared__ unsigned long long s_best;
    __shared__ int s_last;
    constexpr int NW = kTopkThreads / kWarp;
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid / kWarp;
    const int B = p.B, G = (int)gridDim.x;
    const int b = (int)blockIdx.x % B, r = (int)blockIdx.x / B;
    const int g = (G - b + B - 1) / B;   // CTAs serving row b
    const int hv = p.H >> 3;
    uint4 *hs = dyn;                                                   // [H / 8] the row's hidden state
    uint32_t *keys = reinterpret_cast<uint32_t *>(dyn + hv);           // [C] score keys
    int32_t *sel = reinterpret_cast<int32_t *>(keys + p.C);            // [K] selected centroids
    int32_t *clo = sel + p.K;                                          // [K] their first positions
    int32_t *pre = clo + p.K;                                          // [K + 1] candidates before each
    if (tid == 0) s_best = 0ull;
    topk_clear(ts);
    // the candidates' token ids (and ranges) are looked up right after the selection
    prefetch_l2_table(p.ordering, (size_t)p.V * sizeof(int32_t));
    prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    // the scores come from the projection kernel before this one (and the hidden rows,
    // with host-resident input, from the staging kernel before that)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < hv; i += kTopkThreads) hs[i] = ld_ro16(p.hidden + (size_t)b * p.H + (size_t)i * 8);
    select_topk_row(p.scores + (size_t)b * p.C, p.C, p.K, p.bf16_scores != 0, keys, sel, nullptr, ts);

    // the row's candidates: selected clusters (of this shard) in selection order
    if (p.K <= kWarp) {
        // one warp: sizes, then a warp-wide prefix
        if (warp == 0) {
            int lo = 0, hi = 0;
            if (lane < p.K) {
                const int c = sel[lane];
                if (c >= p.c_begin && c < p.c_end) cluster_range(p.offsets, p.V, p.S, c, &lo, &hi, p.ctrl + kCtrlError);
            }
            const int sz = hi - lo;
            int incl = sz;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < p.K) {
                clo[lane] = lo;
                pre[lane] = incl - sz;
            }
            if (lane == p.K - 1) pre[p.K] = incl;
        }
        __syncthreads();
    } else {
        const int per = (p.K + kTopkThreads - 1) / kTopkThreads;
        const int i0 = min(p.K, tid * per), i1 = min(p.K, i0 + per);
        int cnt = 0;
        for (int i = i0; i < i1; ++i) {
            const int c = sel[i];
            int lo = 0, hi = 0;
            if (c >= p.c_begin && c < p.c_end) cluster_range(p.offsets, p.V, p.S, c, &lo, &hi, p.ctrl + kCtrlError);
            clo[i] = lo;
            pre[i] = hi - lo;
            cnt += hi - lo;
        }
        int total;
        int run = cta_exclusive_scan(cnt, ts.scan, &total);
        for (int i = i0; i < i1; ++i) {
            const int sz = pre[i];
            pre[i] = run;
            run += sz;
        }
        if (tid == 0) pre[p.K] = total;
        __syncthreads();
    }
    const long long N = pre[p.K];
    const int s0 = (int)(N * r / g), s1 = (int)(N * (r + 1) / g);
    const int w0 = s0 + (int)((long long)(s1 - s0) * warp / NW);
    const int w1 = s0 + (int)((long long)(s1 - s0) * (warp + 1) / NW);

    // token id of the row's candidate idx (this lane's), -1 past the warp's part or
    // for an id outside [0, V) (reported, skipped)
    auto lane_token = [&](int idx) -> int {
        if (idx >= w1) return -1;
        int lo = 0, hi = p.K;   // pre[lo] <= idx < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= idx) lo = mid;
            else hi = mid;
        }
        const int tok = __ldg(p.ordering + clo[lo] + (idx - pre[lo]));
        if ((unsigned)tok >= (unsigned)p.V) {
            atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
            return -1;
        }
        return tok;
    };

    unsigned long long best = 0ull;
    auto finish = [&](const uint4 (&e)[NCH], int tok) {
        float acc = dot_row<NCH>(e, hs, hv, lane);
        if (p.bf16_logits) acc = round_bf16(acc);
        if (SCATTER) {
            if (lane == 0) p.out_logits[(size_t)b * p.V + tok] = acc;
        } else {
            const unsigned long long k = argmax_key(acc, tok);
            best = k > best ? k : best;
        }
    };

    // Batches of R consecutive candidates, two batches in flight per warp: batch a holds
    // candidates k .. k+R-1 while batch b (the next R) loads.  Short rows take larger
    // batches, so that a warp keeps about as many bytes in flight whatever H.
    constexpr int R = select_gather_batch(NCH);
    uint4 ea[R][NCH], eb[R][NCH];
    int ta[R], tb[R];
    int base = w0;
    int mytok = lane_token(w0 + lane);
    auto token_of = [&](int k) -> int {   // warp-uniform k, called in order; refills per 32
        if (k - base == kWarp) {
            base = k;
            mytok = lane_token(base + lane);
        }
        return __shfl_sync(0xffffffffu, mytok, k - base);
    };
    auto load_batch = [&](uint4 (&e)[R][NCH], int (&t)[R], int k) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            t[i] = k + i < w1 ? token_of(k + i) : -1;
            if (t[i] >= 0) load_row<NCH>(e[i], p.embed + (size_t)t[i] * p.ld, hv, lane);
        }
    };
    auto finish_batch = [&](const uint4 (&e)[R][NCH], const int (&t)[R]) {
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (t[i] >= 0) finish(e[i], t[i]);
    };
    if (w0 < w1) load_batch(ea, ta, w0);
    for (int k = w0; k < w1; k += 2 * R) {
        if (k + R < w1) load_batch(eb, tb, k + R);
        finish_batch(ea, ta);
        if (k + R >= w1) break;
        if (k + 2 * R < w1) load_batch(ea, ta, k + 2 * R);
        finish_batch(eb, tb);
    }
    if (SCATTER) return;

    if (lane == 0 && best) atomicMax(&s_best, best);
    __syncthreads();
    // the CTA's best key of its row, then the ticket (whose release orders the key before
    // it): the last CTA to finish turns the keys into token ids
    if (tid == 0) {
        if (s_best) red_max_u64(p.keys + b, s_best);
        s_last = atom_add_acq_rel(p.ctrl + kCtrlTicket, 1u) == (unsigned)G - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    for (int i = tid; i < B; i += kTopkThreads) {
        const unsigned long long k = atomicAdd(p.keys + i, 0ull);
        int32_t t;
        float v;
        decode_argmax_key(k, &t, &v);
        p.out_tokens[i] = t;
        if (p.out_max) p.out_max[i] = v;
    }
}

size_t select_gather_smem(const GatherParams &p)
{
    return (size_t)(p.H / 8) * sizeof(uint4) + (size_t)p.C * sizeof(uint32_t) +
           (size_t)(3 * p.K + 1) * sizeof(int32_t);
}

template <int NCH, bool SCATTER>
cudaError_t run_select_gather(const GatherParams &p, cudaStream_t s)
{
    const size_t smem = select_gather_smem(p);
    const void *fn = (const void *)k_select_gather<NCH, SCATTER>;
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess) return e;
    const int want = p.B >= 2 && p.H <= 1536 ? kSelectGatherCtasPerSmShort : kSelectGatherCtasPerSm;
    const int per_sm = std::max(1, std::min(want, blocks_per_sm(fn, kTopkThreads, smem)));
    const int grid = std::max(p.B, per_sm * sm_count());
    return launch_dependent(k_select_gather<NCH, SCATTER>, dim3((unsigned)grid), dim3(kTopkThreads), smem, s, p);
}

template <bool SCATTER>
cudaError_t dispatch_select_gather(const GatherParams &p, cudaStream_t s)
{
    switch (chunks_for_hidden(p.H)) {
    case 1: return run_select_gather<1, SCATTER>(p, s);
    case 2: return run_select_gather<2, SCATTER>(p, s);
    case 3: return run_select_gather<3, SCATTER>(p, s);
    case 4: return run_select_gather<4, SCATTER>(p, s);
    case 5: return run_select_gather<5, SCATTER>(p, s);
    case 6: return run_select_gather<6, SCATTER>(p, s);
    case 8: return run_select_gather<8, SCATTER>(p, s);
    case 10: return run_select_gather<10, SCATTER>(p, s);
    case 12: return run_select_gather<12, SCATTER>(p, s);
    case 16: return run_select_gather<16, SCATTER>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_select_gather(const GatherParams &p, bool scatter, cudaStream_t s)
{
    if (p.B < 1 || p.K < 1 || p.K > kSelectGatherMaxK || p.sparse_width || !p.scores) return cudaErrorInvalidValue;
    return scatter ? dispatch_select_gather<true>(p, s) : dispatch_select_gather<false>(p, s);
}

}  // namespace mtp
