// Device helpers and launch parameters shared by the head's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp_head.h"

namespace mtp {

constexpr int kWarp = 32;

// Workspace control words (uint32 at the start of the workspace).
constexpr int kCtrlError = 0;    // MTP_DEVERR_* bits
constexpr int kCtrlItems = 1;    // number of gather work items built by the top-K kernel
constexpr int kCtrlTicket = 2;   // CTAs of the gather-score kernel that have finished
constexpr int kCtrlNext = 3;     // the gathers' item counter: items handed out after the first round
constexpr int kCtrlWaitSite = 4; // first wait that gave up: site code (see score.cu)
constexpr int kCtrlWaitCta = 5;  //   its CTA
constexpr int kCtrlWaitSeq = 6;  //   its slot sequence number or h-buffer use
constexpr int kCtrlWords = 16;

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------

// 16-byte read-only load that bypasses L1 (rows are read once) and asks L2 to
// fetch the surrounding 256 bytes (embedding rows are long contiguous runs).
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 16-byte read-only load through the normal cache path (small, reused data).
__device__ __forceinline__ uint4 ld_ro16(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// L2 prefetch hint for a small read-only table (token ordering, cluster offsets) that a
// gather kernel reads on the dependent chain of every work item: issued before the
// kernel waits for the previous kernel of the call, so the table is in L2 by the time
// the work items arrive.  The grid's threads take one 128-byte step of the table each;
// every address lies inside it.
__device__ __forceinline__ void prefetch_l2_table(const void *base, size_t bytes)
{
    if (base == nullptr) return;
    const size_t nthreads = (size_t)gridDim.x * blockDim.x;
    for (size_t off = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 128; off < bytes; off += nthreads * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"((const char *)base + off));
}

// ---------------------------------------------------------------------------
// bf16 arithmetic: a bf16 is the top half of an fp32, so unpacking is a shift
// or a mask; products of two bf16 values are exact in fp32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// acc + sum of the 8 products of two 16-byte groups of bf16 values.
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b, float acc)
{
    acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
    acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
    acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
    acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
    acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
    acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
    acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
    acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
    return acc;
}

// The same sum with f32 FMAs that take the bf16 halves directly (sm_100 family):
// products are exact and each step rounds once, so the result is bit-identical
// to dot8_bf16 while skipping the unpacking instructions.
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float acc)
{
    asm("{\n"
        " .reg .b16 a0, a1, b0, b1;\n"
        " mov.b32 {a0, a1}, %1;\n"
        " mov.b32 {b0, b1}, %2;\n"
        " fma.rn.f32.bf16 %0, a0, b0, %0;\n"
        " fma.rn.f32.bf16 %0, a1, b1, %0;\n"
        "}\n"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

__device__ __forceinline__ float dot8_bf16_mixed(uint4 a, uint4 b, float acc)
{
    acc = fma2_bf16(a.x, b.x, acc);
    acc = fma2_bf16(a.y, b.y, acc);
    acc = fma2_bf16(a.z, b.z, acc);
    acc = fma2_bf16(a.w, b.w, acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Order-preserving keys
// ---------------------------------------------------------------------------

// fp32 -> uint32 whose unsigned order is the float order; -0 and +0 map to
// the same key.
__device__ __forceinline__ uint32_t ord_key(float f)
{
    f = __fadd_rn(f, 0.0f);  // -0 -> +0
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// v rounded to the nearest bf16 value (ties to even), as an fp32 value.
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ float ord_value(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// 64-bit argmax key: larger logit wins, then lower token id.  Never 0 for a
// finite logit, so 0 means "no candidate".
__device__ __forceinline__ unsigned long long argmax_key(float v, int32_t token)
{
    return ((unsigned long long)ord_key(v) << 32) |
           (unsigned long long)(0xffffffffu - (uint32_t)token);
}

__device__ __forceinline__ void decode_argmax_key(unsigned long long k, int32_t *token, float *v)
{
    if (k == 0ull) {
        *token = -1;
        *v = __int_as_float(0xff800000);  // -inf
    } else {
        *token = (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
        *v = ord_value((uint32_t)(k >> 32));
    }
}

// Fire-and-forget 64-bit max at device scope (no ordering of its own; a later release
// operation of the same thread orders it).
__device__ __forceinline__ void red_max_u64(unsigned long long *addr, unsigned long long v)
{
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

// atomicAdd with acquire-release semantics at device scope: the thread's earlier writes
// (and reductions) are visible to whoever acquires a later value of *addr, and this
// thread sees what the earlier adders released.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *addr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// Ordered positions [lo, hi) of centroid c; false (and the error bit) when the
// offsets are malformed.
__device__ __forceinline__ bool cluster_range(const int32_t *offsets, int32_t V, int32_t S, int c,
                                              int *lo, int *hi, uint32_t *err_word)
{
    if (offsets == nullptr) {
        *lo = c * S;
        *hi = *lo + S;
        return true;
    }
    int a = __ldg(offsets + c), b = __ldg(offsets + c + 1);
    if (a < 0 || b < a || b > V) {
        if (err_word) atomicOr(err_word, MTP_DEVERR_OFFSETS);
        *lo = *hi = 0;
        return false;
    }
    *lo = a;
    *hi = b;
    return true;
}

// ---------------------------------------------------------------------------
// Launch parameters
// ---------------------------------------------------------------------------
struct ProjParams {
    const uint16_t *hidden;  // [B, H]
    const uint16_t *wc;      // [C, H]
    float *scores;           // [B, C]
    uint32_t *zero;          // words to clear before the top-K kernel runs (may be null)
    int zero_words;
    int B, H, C;
    int rows_per_group;      // hidden rows staged in shared memory at a time
    int after_fill;          // launched behind the scatter's fill, overlapping it
    int after_stage;         // launched behind the staging of host-resident hidden rows:
                             // reads them only after griddepcontrol.wait
};

struct TopkParams {
    const float *scores;     // [B, C]
    int32_t *topk;           // [B, K] out, sorted by (score desc, index asc)
    int B, C, K, V, S;
    const int32_t *offsets;  // [C+1] or null (uniform clusters of S)
    // bucketing (null rowmask = no bucketing)
    uint32_t *rowmask;       // [C, W] bit b%32 of word b/32: row b selected c
    int W;
    int32_t *ccount;         // [C] rows that selected c
    int2 *items;             // (centroid, first position offset) work items
    int items_cap;           // capacity of items
    uint32_t *ctrl;
    int chunk;               // tokens per work item
    int c_begin, c_end;      // clusters this shard gathers (bucketing skips the others)
    int bf16_scores;         // select on the scores rounded to bf16
};

struct GatherParams {
    const uint16_t *hidden;         // [B, H]
    const uint16_t *embed;          // [>=V, ld]
    const uint8_t *packed;          // packed embedding table (tensor-core gather), or null
    int packed_clusters;            // clusters the packed table was sized for (its shard)
    long long ld;
    const int32_t *ordering;        // [V]
    const int32_t *offsets;         // [C+1] or null
    const uint32_t *rowmask;        // [C, W]
    const int2 *items;
    int items_cap;
    uint32_t *ctrl;
    unsigned long long *keys;       // [B] argmax keys (argmax finish)
    float *out_logits;              // [B, V] (scatter finish)
    int32_t *out_tokens;            // [B] (argmax finish)
    float *out_max;                 // [B] or null
    // the sparse pair (scatter instantiation): out_logits / out_ids are [B, sparse_width]
    // with sparse_width = K * S, entry (row, rank k of the cluster in the row's top-K,
    // position i in the cluster) at row * sparse_width + k * S + i; 0 = full-vocab scatter
    int sparse_width;
    int32_t *out_ids;               // [B, sparse_width] or null
    const int32_t *topk;            // [B, K] the rows' selections (ranks for the sparse pair)
    int K;
    int bf16_logits;                // round every logit to bf16 before storing or comparing it
    int B, H, V, S, W, C;
    int chunk;                      // ordered positions per work item
    int ring;                       // embedding-row slots per CTA
    int row_group;                  // hidden rows per h buffer
    int step;                       // slots the producer warp publishes per batch (<= 32, <= ring)
    int consumer_warps;             // 8 or 16
    int ctas_per_sm;                // gather CTAs per SM (1 or 2)
    // the fused small-batch kernel selects each row's top-K itself
    const float *scores;            // [B, C] centroid scores
    int bf16_scores;                // select on the scores rounded to bf16
    int c_begin, c_end;             // clusters this shard gathers
    // bounded waits of the pipelined gather: wall-clock limit, and the wait test (its
    // first h-buffer wait waits for a barrier phase that nothing completes)
    unsigned long long wait_ns;
    int stall_test;
};

}  // namespace mtp
