// Centroid projection: scores[b, c] = sum_k hidden[b, k] * Wc[c, k].
//
// Step 1 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): the
// bias-free centroid Linear applied to the draft hidden states.  Here it is
// accumulated in fp32 from the bf16 inputs and kept in fp32.
//
// CUDA-core form for small batches: each warp holds two centroid rows in
// registers (one 16-byte load per lane per 256 elements) and dots them with the
// hidden rows, which the CTA stages in shared memory a group at a time, R rows at
// once (2R independent sums per lane, reduced together; R = 1, 2, 4 or 8 by the
// batch, each its own instantiation, the last rows of a group padded).  Wc
// is read from HBM exactly once per call.  The same kernel clears the
// workspace's control region for the kernels that follow it on the stream.
#include "internal.h"

namespace mtp {

// Scores of the staged hidden rows r0 .. r0 + R - 1 (rows row0 .. of the batch; only the
// first nr are real, the others padding whose sums are dropped) against
// this warp's centroid rows c0, c0 + 1: each lane's partial dot products of the 2R
// (row, centroid) pairs, then one reduce-scatter butterfly over the warp: at each xor
// step a lane keeps half of its values and adds its partner's copies of them, so the
// offsets 16, 8, ... leave every value's sum on a pair or group of lanes after 2R
// shuffles (one warp_sum per value would take 10R).  The additions are warp_sum's, in
// its order (xor 16 first), so the scores are the same bits.
template <int NCH, int R>
__device__ __forceinline__ void proj_rows(const ProjParams &p, const uint4 (&w0)[NCH], const uint4 (&w1)[NCH],
                                          const uint4 *hs, int hv, int lane, int r0, int row0, int nr, int c0,
                                          bool v1)
{
    constexpr int V = 2 * R;
    constexpr int kSteps = V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : 4;
    static_assert(V == 1 << kSteps, "R is 1, 2, 4 or 8");
    float a[V];
#pragma unroll
    for (int j = 0; j < V; ++j) a[j] = 0.f;
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int idx = k * kWarp + lane;
        if (idx < hv) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 x = hs[(r0 + r) * hv + idx];
                a[2 * r] = dot8_bf16(w0[k], x, a[2 * r]);
                a[2 * r + 1] = dot8_bf16(w1[k], x, a[2 * r + 1]);
            }
        }
    }
    int vi = 0;   // the value (2 * row + centroid) whose sum this lane ends with
#pragma unroll
    for (int h = V / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? a[i] : a[i + h];
            const float keep = up ? a[i + h] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) vi += h;
    }
#pragma unroll
    for (int o = 16 >> kSteps; o >= 1; o >>= 1) a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
    if ((lane & ((32 >> kSteps) - 1)) == 0) {   // one lane per value
        const int cen = vi & 1;
        if ((vi >> 1) < nr && (!cen || v1)) p.scores[(size_t)(row0 + (vi >> 1)) * p.C + c0 + cen] = a[0];
    }
}

template <int NCH, int R>
__global__ void __launch_bounds__(kProjThreads) k_projection(ProjParams p)
{
    extern __shared__ uint4 hs[];  // [rows_per_group rounded up to R][H / 8]
    const int tid = threadIdx.x;
    // let the next kernel of the call (the top-K) be scheduled now; it waits for our results
    asm volatile("griddepcontrol.launch_dependents;");
    for (int i = blockIdx.x * kProjThreads + tid; i < p.zero_words; i += gridDim.x * kProjThreads)
        p.zero[i] = 0u;

    const int lane = tid & (kWarp - 1), warp = tid / kWarp;
    const int hv = p.H >> 3;
    const int c0 = (blockIdx.x * (kProjThreads / kWarp) + warp) * kProjRowsPerWarp;
    const bool v0 = c0 < p.C, v1 = c0 + 1 < p.C;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

    uint4 w0[NCH], w1[NCH];
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        const int idx = k * kWarp + lane;
        const bool in = idx < hv;
        w0[k] = (in && v0) ? ld_stream16(p.wc + (size_t)c0 * p.H + idx * 8) : zero;
        w1[k] = (in && v1) ? ld_stream16(p.wc + (size_t)(c0 + 1) * p.H + idx * 8) : zero;
    }

    // launched behind the kernel that stages host-resident hidden rows: the centroid
    // rows above are already streaming; the hidden rows are read only once it is done
    if (p.after_stage) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int b0 = 0; b0 < p.B; b0 += p.rows_per_group) {
        const int nb = min(p.rows_per_group, p.B - b0);
        __syncthreads();  // previous group fully consumed
        const uint16_t *src = p.hidden + (size_t)b0 * p.H;
        for (int i = tid; i < nb * hv; i += kProjThreads)
            hs[i] = ld_ro16(src + (size_t)i * 8);
        __syncthreads();
        if (!v0)
            continue;
        for (int r = 0; r < nb; r += R) proj_rows<NCH, R>(p, w0, w1, hs, hv, lane, r, b0 + r, min(R, nb - r), c0, v1);
    }
    // launched behind the scatter's fill (which it does not read): complete only after it
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int NCH, int R>
static cudaError_t run_projection_r(const ProjParams &p, cudaStream_t s)
{
    // the padding rows of the last group of R read staged memory (whatever it holds)
    const size_t smem = (size_t)((p.rows_per_group + R - 1) / R * R) * p.H * sizeof(uint16_t);
    const void *fn = (const void *)k_projection<NCH, R>;
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    const int rows_per_cta = (kProjThreads / kWarp) * kProjRowsPerWarp;
    const int grid = (p.C + rows_per_cta - 1) / rows_per_cta;
    if (p.after_fill || p.after_stage)
        return launch_dependent(k_projection<NCH, R>, dim3(grid), dim3(kProjThreads), smem, s, p);
    k_projection<NCH, R><<<grid, kProjThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// Rows reduced together: the batch's rows (per staged group) up to 8, a power of two.
template <int NCH>
static cudaError_t run_projection(const ProjParams &p, cudaStream_t s)
{
    const int rows = p.rows_per_group < p.B ? p.rows_per_group : p.B;
    if (rows >= 5) return run_projection_r<NCH, 8>(p, s);
    if (rows >= 3) return run_projection_r<NCH, 4>(p, s);
    if (rows == 2) return run_projection_r<NCH, 2>(p, s);
    return run_projection_r<NCH, 1>(p, s);
}

cudaError_t launch_projection(const ProjParams &p, cudaStream_t s)
{
    switch (chunks_for_hidden(p.H)) {
    case 1: return run_projection<1>(p, s);
    case 2: return run_projection<2>(p, s);
    case 3: return run_projection<3>(p, s);
    case 4: return run_projection<4>(p, s);
    case 5: return run_projection<5>(p, s);
    case 6: return run_projection<6>(p, s);
    case 8: return run_projection<8>(p, s);
    case 10: return run_projection<10>(p, s);
    case 12: return run_projection<12>(p, s);
    case 16: return run_projection<16>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mtp
