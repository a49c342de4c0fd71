// Gather + sparse dot products + argmax / scatter, and the dense comparator.
//
// Steps 3-4 and the two finishes of Gemma4MTPMaskedEmbedder ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py):
// _select_and_score maps each selected centroid to its token ids through
// token_ordering.view(C, V/C), gathers those lm_head rows and dots them with
// the hidden state; get_top_tokens keeps the token id of the largest logit;
// forward scatters the logits into a full-vocabulary row that is -inf
// elsewhere (the -inf fill is a separate kernel that runs first).
//
// Work is cluster-major: a work item is a chunk of one selected cluster's
// ordered positions together with every batch row that selected the cluster
// (the bucket built by the top-K kernel).  Each candidate embedding row is
// therefore read from HBM once per call however many rows picked its
// cluster.  A warp takes two candidate rows at a time, loads each with
// 16-byte loads (512 contiguous bytes per warp instruction), and dots them
// against the bucket's hidden rows staged in shared memory; a butterfly of
// shuffles finishes each dot product.  Argmax keys (logit, lower token id)
// are combined with a 64-bit atomicMax per row, and the last CTA to finish
// turns them into token ids, so no grid-wide wait is ever needed.
//
// Dense mode reuses the loop over every token in id order with every batch
// row (the comparator head).
#include "internal.h"

namespace mtp {

template <int NCH, int MODE>
__global__ void __launch_bounds__(kScoreThreads) k_gather_score(ScoreParams p)
{
    extern __shared__ uint4 hs[];             // [rows_per_group][H / 8]
    __shared__ int s_rows[MTP_MAX_BATCH];     // batch rows of the current item
    __shared__ int s_item, s_nrows, s_last;

    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid / kWarp;
    const int hv = p.H >> 3;
    const bool want_keys = p.keys != nullptr;
    const bool want_logits = p.out_logits != nullptr;
    const int n_items = (MODE == kDense) ? p.dense_items : (int)min(p.ctrl[kCtrlItems], (uint32_t)p.items_cap);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

    for (int round = 0;; ++round) {
        int it;
        if (MODE == kDense) {
            it = blockIdx.x + round * gridDim.x;
        } else {
            // dynamic hand-out: items differ in size (ragged clusters, bucket sizes)
            if (tid == 0) s_item = (int)atomicAdd(p.ctrl + kCtrlNext, 1u);
            __syncthreads();
            it = s_item;
        }
        if (it >= n_items)
            break;

        int pbeg, pend, nrows;
        if (MODE == kDense) {
            pbeg = it * p.chunk;
            pend = min(p.V, pbeg + p.chunk);
            nrows = p.B;
        } else {
            int2 item = p.items[it];
            int lo = 0, hi = 0;
            // items are written by the top-K kernel; the checks only matter when malformed
            // offsets made it drop some (then a slot may hold an earlier call's item)
            if ((unsigned)item.x >= (unsigned)p.C || item.y < 0) item = make_int2(0, 0x7fffffff);
            cluster_range(p.offsets, p.V, p.S, item.x, &lo, &hi, nullptr);
            pbeg = (item.y > hi - lo) ? hi : lo + item.y;
            pend = min(hi, pbeg + p.chunk);
            if (warp == 0) {
                uint32_t w = lane < p.W ? p.rowmask[(size_t)item.x * p.W + lane] : 0u;
                const int cnt = __popc(w);
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < kWarp; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                int pos = incl - cnt;
                while (w) {
                    const int bit = __ffs(w) - 1;
                    s_rows[pos++] = lane * kWarp + bit;
                    w &= w - 1u;
                }
                if (lane == kWarp - 1) s_nrows = incl;
            }
            __syncthreads();
            nrows = s_nrows;
        }

        for (int g0 = 0; g0 < nrows; g0 += p.rows_per_group) {
            const int gr = min(p.rows_per_group, nrows - g0);
            for (int i = tid; i < gr * hv; i += kScoreThreads) {
                const int r = i / hv, k = i - r * hv;
                const int row = (MODE == kDense) ? g0 + r : s_rows[g0 + r];
                hs[i] = ld_ro16(p.hidden + (size_t)row * p.H + (size_t)k * 8);
            }
            __syncthreads();

            // lane r keeps the running best of the group's r-th row
            const int my_row = lane < gr ? ((MODE == kDense) ? g0 + lane : s_rows[g0 + lane]) : 0;
            unsigned long long best = 0ull;

            for (int pa = pbeg + warp; pa < pend; pa += 2 * kScoreWarps) {
                const int pb = pa + kScoreWarps;
                const bool has_b = pb < pend;
                int ta, tb;
                if (MODE == kDense) {
                    ta = pa;
                    tb = pb;
                } else {
                    ta = __ldg(p.ordering + pa);
                    tb = has_b ? __ldg(p.ordering + pb) : 0;
                }
                const bool ok_a = (unsigned)ta < (unsigned)p.V;
                const bool ok_b = has_b && (unsigned)tb < (unsigned)p.V;
                if (MODE != kDense && lane == 0 && (!ok_a || (has_b && !ok_b)))
                    atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
                const uint16_t *ra = p.embed + (long long)(ok_a ? ta : 0) * p.ld;
                const uint16_t *rb = p.embed + (long long)(ok_b ? tb : 0) * p.ld;

                uint4 ea[NCH], eb[NCH];
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    const int idx = k * kWarp + lane;
                    const bool in = idx < hv;
                    ea[k] = (in && ok_a) ? ld_stream16(ra + idx * 8) : zero;
                    eb[k] = (in && ok_b) ? ld_stream16(rb + idx * 8) : zero;
                }
                for (int r = 0; r < gr; ++r) {
                    float sa = 0.f, sb = 0.f;
#pragma unroll
                    for (int k = 0; k < NCH; ++k) {
                        const int idx = k * kWarp + lane;
                        if (idx < hv) {
                            const uint4 x = hs[r * hv + idx];
                            sa = dot8_bf16(ea[k], x, sa);
                            sb = dot8_bf16(eb[k], x, sb);
                        }
                    }
                    sa = warp_sum(sa);
                    sb = warp_sum(sb);
                    if (lane == r) {
                        if (want_keys) {
                            if (ok_a) best = max(best, argmax_key(sa, ta));
                            if (ok_b) best = max(best, argmax_key(sb, tb));
                        }
                        if (want_logits) {
                            float *orow = p.out_logits + (size_t)my_row * p.V;
                            if (ok_a) orow[ta] = sa;
                            if (ok_b) orow[tb] = sb;
                        }
                    }
                }
            }
            if (want_keys && lane < gr && best != 0ull)
                atomicMax(p.keys + my_row, best);
            __syncthreads();  // hs and s_rows are rewritten next
        }
    }

    if (!want_keys)
        return;
    // Last CTA to finish decodes the per-row keys (threadfence-reduction pattern).
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(p.ctrl + kCtrlTicket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    for (int b = tid; b < p.B; b += kScoreThreads) {
        const unsigned long long k = atomicAdd(p.keys + b, 0ull);
        int32_t tok;
        float v;
        decode_argmax_key(k, &tok, &v);
        p.out_tokens[b] = tok;
        if (p.out_max) p.out_max[b] = v;
    }
}

template <int NCH, int MODE>
static cudaError_t run_score(const ScoreParams &p, cudaStream_t s, int *grid_out)
{
    const size_t smem = (size_t)p.rows_per_group * p.H * sizeof(uint16_t);
    const void *fn = (const void *)k_gather_score<NCH, MODE>;
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = blocks_per_sm(fn, kScoreThreads, smem);
    if (per_sm < 1) per_sm = 1;
    int grid = sm_count() * per_sm;
    if (MODE == kDense && grid > p.dense_items) grid = p.dense_items;
    if (grid < 1) grid = 1;
    *grid_out = grid;
    k_gather_score<NCH, MODE><<<grid, kScoreThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t dispatch_score(const ScoreParams &p, cudaStream_t s, int *grid)
{
    switch (chunks_for_hidden(p.H)) {
    case 1: return run_score<1, MODE>(p, s, grid);
    case 2: return run_score<2, MODE>(p, s, grid);
    case 3: return run_score<3, MODE>(p, s, grid);
    case 4: return run_score<4, MODE>(p, s, grid);
    case 5: return run_score<5, MODE>(p, s, grid);
    case 6: return run_score<6, MODE>(p, s, grid);
    case 8: return run_score<8, MODE>(p, s, grid);
    case 10: return run_score<10, MODE>(p, s, grid);
    case 12: return run_score<12, MODE>(p, s, grid);
    case 16: return run_score<16, MODE>(p, s, grid);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_score(const ScoreParams &p, ScoreMode mode, cudaStream_t s, int *grid)
{
    return mode == kDense ? dispatch_score<kDense>(p, s, grid)
                          : dispatch_score<kMaskedArgmax>(p, s, grid);
}

// forward's fill: every entry of the [B, V] row block is -inf before the
// scatter writes the candidates' logits.
__global__ void __launch_bounds__(256) k_fill_neg_inf(float *out, size_t n)
{
    const float ninf = __int_as_float(0xff800000);
    const float4 v = make_float4(ninf, ninf, ninf, ninf);
    float4 *o4 = reinterpret_cast<float4 *>(out);
    const size_t n4 = n / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x)
        o4[i] = v;
    if (blockIdx.x == 0 && threadIdx.x < (n & 3))
        out[n4 * 4 + threadIdx.x] = ninf;
}

cudaError_t launch_fill_neg_inf(float *out, size_t n, cudaStream_t s)
{
    const int per_sm = blocks_per_sm((const void *)k_fill_neg_inf, 256, 0);
    const int grid = sm_count() * (per_sm > 0 ? per_sm : 1);
    k_fill_neg_inf<<<grid, 256, 0, s>>>(out, n);
    return cudaGetLastError();
}

}  // namespace mtp
