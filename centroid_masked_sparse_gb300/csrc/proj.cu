// Centroid projection: scores[b, c] = sum_k hidden[b, k] * Wc[c, k].
//
// Step 1 of Gemma4MTPMaskedEmbedder._select_and_score ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py): the
// bias-free centroid Linear applied to the draft hidden states.  Here it is
// accumulated in fp32 from the bf16 inputs and kept in fp32.
//
// CUDA-core form for every batch: each warp holds two centroid rows in
// registers (one 16-byte load per lane per 256 elements) and dots them with the
// hidden rows, which the CTA stages in shared memory a group at a time.  Wc is
// read from HBM exactly once per call.  The same kernel clears the
// workspace's control region for the kernels that follow it on the stream.
#include "internal.h"

namespace mtp {

template <int NCH>
__global__ void __launch_bounds__(kProjThreads) k_projection(ProjParams p)
{
    extern __shared__ uint4 hs[];  // [rows_per_group][H / 8]
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
        for (int r = 0; r < nb; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
                const int idx = k * kWarp + lane;
                if (idx < hv) {
                    const uint4 x = hs[r * hv + idx];
                    a0 = dot8_bf16(w0[k], x, a0);
                    a1 = dot8_bf16(w1[k], x, a1);
                }
            }
            a0 = warp_sum(a0);
            a1 = warp_sum(a1);
            if (lane == 0) {
                float *row = p.scores + (size_t)(b0 + r) * p.C;
                row[c0] = a0;
                if (v1)
                    row[c0 + 1] = a1;
            }
        }
    }
    // launched behind the scatter's fill (which it does not read): complete only after it
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int NCH>
static cudaError_t run_projection(const ProjParams &p, cudaStream_t s)
{
    const size_t smem = (size_t)p.rows_per_group * p.H * sizeof(uint16_t);
    const void *fn = (const void *)k_projection<NCH>;
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess)
        return e;
    const int rows_per_cta = (kProjThreads / kWarp) * kProjRowsPerWarp;
    const int grid = (p.C + rows_per_cta - 1) / rows_per_cta;
    if (p.after_fill || p.after_stage)
        return launch_dependent(k_projection<NCH>, dim3(grid), dim3(kProjThreads), smem, s, p);
    k_projection<NCH><<<grid, kProjThreads, smem, s>>>(p);
    return cudaGetLastError();
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
