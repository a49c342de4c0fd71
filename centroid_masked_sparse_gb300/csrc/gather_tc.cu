// Gather + sparse dot products on the tensor cores, for calls whose buckets are
// large (many batch rows chose the same cluster).
//
// Steps 3-4 and both finishes of Gemma4MTPMaskedEmbedder ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py), like
// score.cu, but each work item is treated as the dense contraction it is when
// its bucket holds many rows: logits[t, r] = sum_k E[tok_t, k] * h[row_r, k] for
// the item's ≤128 candidate positions t and the bucket's rows r.
//
// One unit = (work item, block of ≤128 bucket rows).  The candidate embedding
// rows are the MMA's M side (one token per TMEM lane), the bucket's hidden rows
// its N side (padded to a multiple of 16 per unit), K = H in 64-element blocks.
// Both operands are gathered by TMA with tile::gather4 (four arbitrary rows of
// 64 bf16 per instruction, 128-byte swizzle, the layout the MMA descriptors
// expect); padding rows use an out-of-range row coordinate, which TMA fills
// with zeros without reading memory.  With the cluster-ordered copy of the
// embedding table the item's candidate rows are consecutive, and the A tile is
// one plain 64 x 128 TMA tile load instead of 32 gathers (rows past the
// cluster's end are loaded but their lanes are ignored).  Warp roles per CTA
// (one CTA per SM):
//   warp 4   producer: per unit, builds the token and row lists in a small
//            metadata ring, then per k-block lets each lane issue one gather4 of
//            candidate rows (and of hidden rows) into a ring of stages;
//   warp 5   one thread issues tcgen05.mma (kind::f16, fp32 in TMEM,
//            double-buffered accumulators);
//   warps 0-3 epilogue: tcgen05.ld of the unit's logits (thread = candidate),
//            then the scatter store or the per-row argmax fold.
// Every mbarrier wait is bounded and records MTP_DEVERR_TIMEOUT if it gives up.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace mtp {

using namespace sm100;

namespace {

constexpr int kThreads = 192;
constexpr int kTileM = 128;        // candidate positions per unit
constexpr int kTileK = 64;         // bf16 per k-block (128-byte rows)
constexpr int kMaxN = 128;         // bucket rows per unit
constexpr int kMeta = 4;           // unit-metadata ring
constexpr uint32_t kABytes = kTileM * kTileK * 2;
constexpr uint64_t kWaitNs = 2000000000ull;

struct UnitMeta {
    int tok[kTileM];    // candidate token ids (-1: padding)
    int rows[kMaxN];    // bucket rows of this unit (n of them)
    int n, npad, nvalid, pad;
};

struct Params {
    const int32_t *ordering;
    const int32_t *offsets;
    const uint32_t *rowmask;
    const int2 *items;
    int items_cap;
    uint32_t *ctrl;
    unsigned long long *keys;
    float *out_logits;
    int32_t *out_tokens;
    float *out_max;
    int B, H, V, S, W, C;
    int chunk;      // positions per work item (<= 128)
    int ordered;    // tmap_e is the cluster-ordered table in 64 x 128 tiles
    int num_kb;
    int stages;
};

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int x, int y0, int y1,
                                            int y2, int y3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void timeout(const Params &p)
{
    atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TIMEOUT);
}

// Rows of the bucket of cluster c in row order, block `blk` (kMaxN rows per block):
// the warp writes them to `rows` and returns how many (all lanes).
__device__ int bucket_rows(const Params &p, int c, int blk, int lane, int *rows)
{
    const uint32_t w = lane < p.W ? __ldcg(p.rowmask + (size_t)c * p.W + lane) : 0u;
    const int cnt = __popc(w);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int pos = incl - cnt;
    const int lo = blk * kMaxN, hi = lo + kMaxN;
    for (uint32_t m = w; m; m &= m - 1u, ++pos)
        if (pos >= lo && pos < hi) rows[pos - lo] = lane * kWarp + __ffs(m) - 1;
    const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
    return max(0, min(kMaxN, total - lo));
}

template <bool SCATTER>
__global__ void __launch_bounds__(kThreads, 1)
    k_gather_tc(const __grid_constant__ CUtensorMap tmap_e, const __grid_constant__ CUtensorMap tmap_h,
                const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages;
    constexpr uint32_t kBBytes = kMaxN * kTileK * 2;
    uint8_t *a_smem = smem;
    uint8_t *b_smem = smem + (size_t)S * kABytes;
    UnitMeta *meta = reinterpret_cast<UnitMeta *>(b_smem + (size_t)S * kBBytes);
    unsigned long long *best = reinterpret_cast<unsigned long long *>(meta + kMeta);
    uint64_t *bars = reinterpret_cast<uint64_t *>(best + p.B);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 4 + 2 * kMeta);
    __shared__ int s_last;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x & (kWarp - 1);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8u * S;
    const uint32_t tfull0 = empty0 + 8u * S, tempty0 = tfull0 + 16u;
    const uint32_t mfull0 = tempty0 + 16u, mempty0 = mfull0 + 8u * kMeta;
    constexpr uint32_t kTmemCols = 2 * kMaxN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, 4);
        }
        for (int m = 0; m < kMeta; ++m) {
            mbar_init(mfull0 + 8u * m, 1);
            mbar_init(mempty0 + 8u * m, 5);   // 4 epilogue warps + the MMA thread
        }
        fence_barrier_init();
    }
    if (!SCATTER)
        for (int b = threadIdx.x; b < p.B; b += kThreads) best[b] = 0ull;
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // the work items and buckets come from the top-K kernel before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int n_items = (int)min(p.ctrl[kCtrlItems], (uint32_t)p.items_cap);
    const int G = (int)gridDim.x;
    const int nblk_max = (p.B + kMaxN - 1) / kMaxN;

    if (warp == 4) {
        // ------------------------------------------------------------- producer
        int stage = 0, u = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += G) {
            const int2 item = p.items[it];
            int lo = 0, hi = 0;
            if ((unsigned)item.x < (unsigned)p.C && item.y >= 0)
                cluster_range(p.offsets, p.V, p.S, item.x, &lo, &hi, nullptr);
            const int p0 = item.y > hi - lo ? hi : lo + item.y;
            const int nvalid = max(0, min(min(p.chunk, kTileM), hi - p0));
            if (nvalid == 0) continue;
            for (int blk = 0; blk < nblk_max && ok; ++blk, ++u) {
                const int um = u % kMeta;
                const uint32_t mpar = (uint32_t)(u / kMeta) & 1u;
                if (!mbar_wait(mempty0 + 8u * um, mpar ^ 1u, kWaitNs)) {
                    ok = false;
                    break;
                }
                UnitMeta &m = meta[um];
                const int n = bucket_rows(p, item.x, blk, lane, m.rows);
                if (n == 0) {
                    // no rows in this block (the bucket is smaller): publish an empty unit
                    // so the ring stays in step, then stop this item
                    if (lane == 0) {
                        m.n = 0;
                        m.npad = 0;
                        m.nvalid = 0;
                        __threadfence_block();
                        mbar_arrive(mfull0 + 8u * um);
                    }
                    __syncwarp();
                    ++u;
                    break;
                }
                const int npad = (n + 15) & ~15;
                for (int r = n + lane; r < npad; r += kWarp) m.rows[r] = p.B;   // zero rows
#pragma unroll
                for (int j = 0; j < kTileM / kWarp; ++j) {
                    const int t = j * kWarp + lane;
                    int tok = -1;
                    if (t < nvalid) {
                        tok = __ldg(p.ordering + p0 + t);
                        if ((unsigned)tok >= (unsigned)p.V) {
                            atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
                            tok = -1;
                        }
                    }
                    m.tok[t] = tok;
                }
                if (lane == 0) {
                    m.n = n;
                    m.npad = npad;
                    m.nvalid = nvalid;
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    mbar_arrive(mfull0 + 8u * um);
                }
                // the k-blocks: lane j gathers candidate rows 4j..4j+3 and, while j < npad/4,
                // bucket rows 4j..4j+3 (out-of-range coordinates for padding)
                const int y0 = m.tok[4 * lane] >= 0 ? m.tok[4 * lane] : p.V;
                const int y1 = m.tok[4 * lane + 1] >= 0 ? m.tok[4 * lane + 1] : p.V;
                const int y2 = m.tok[4 * lane + 2] >= 0 ? m.tok[4 * lane + 2] : p.V;
                const int y3 = m.tok[4 * lane + 3] >= 0 ? m.tok[4 * lane + 3] : p.V;
                const bool has_b = 4 * lane < npad;
                const int z0 = has_b ? m.rows[4 * lane] : 0, z1 = has_b ? m.rows[4 * lane + 1] : 0;
                const int z2 = has_b ? m.rows[4 * lane + 2] : 0, z3 = has_b ? m.rows[4 * lane + 3] : 0;
                // candidate groups of four that are all padding are not fetched at all: their
                // tile rows keep stale data, and the epilogue ignores those rows (token -1)
                const bool has_a = 4 * lane < nvalid;
                const uint32_t na = (uint32_t)(nvalid + 3) / 4;
                const uint32_t tx = (p.ordered ? kABytes : na * 4 * 128) + (uint32_t)npad * kTileK * 2;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    int wok = 1;
                    if (lane == 0) {
                        wok = mbar_wait(empty0 + 8u * stage, phase ^ 1u, kWaitNs);
                        if (wok) mbar_arrive_expect_tx(full0 + 8u * stage, tx);
                    }
                    if (!__shfl_sync(0xffffffffu, wok, 0)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = full0 + 8u * stage;
                    if (p.ordered) {
                        if (lane == 0)
                            tma_load_2d(smem_u32(a_smem + (size_t)stage * kABytes), &tmap_e, kb * kTileK, p0, bar);
                    } else if (has_a)
                        tma_gather4(smem_u32(a_smem + (size_t)stage * kABytes + (size_t)lane * 4 * 128),
                                    &tmap_e, kb * kTileK, y0, y1, y2, y3, bar);
                    if (has_b)
                        tma_gather4(smem_u32(b_smem + (size_t)stage * kBBytes + (size_t)lane * 4 * 128),
                                    &tmap_h, kb * kTileK, z0, z1, z2, z3, bar);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (n < kMaxN) {
                    ++u;
                    break;  // the bucket fits this block: no further row block
                }
            }
        }
        // end of stream: an empty unit with n = -1
        if (ok) {
            const int um = u % kMeta;
            const uint32_t mpar = (uint32_t)(u / kMeta) & 1u;
            if (lane == 0) {
                if (mbar_wait(mempty0 + 8u * um, mpar ^ 1u, kWaitNs)) {
                    meta[um].n = -1;
                    __threadfence_block();
                    mbar_arrive(mfull0 + 8u * um);
                } else {
                    ok = false;
                }
            }
        }
        if (!ok && lane == 0) timeout(p);
    } else if (warp == 5) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int u = 0;; ++u) {
                const int um = u % kMeta;
                if (!mbar_wait(mfull0 + 8u * um, (uint32_t)(u / kMeta) & 1u, kWaitNs)) {
                    timeout(p);
                    break;
                }
                const int n = meta[um].n;
                if (n < 0) break;
                const int npad = meta[um].npad;
                mbar_arrive(mempty0 + 8u * um);   // done with this entry's metadata
                if (n == 0) continue;
                if (!mbar_wait(tempty0 + 8u * acc, acc_phase ^ 1u, kWaitNs)) {
                    timeout(p);
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kTileM, npad);
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kMaxN);
                bool ok = true;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(full0 + 8u * stage, phase, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_kmajor_desc(smem_u32(a_smem + (size_t)stage * kABytes));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(b_smem + (size_t)stage * kBBytes));
#pragma unroll
                    for (int k = 0; k < kTileK / 16; ++k)
                        mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(empty0 + 8u * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    timeout(p);
                    break;
                }
                mma_commit(tfull0 + 8u * acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------------------- epilogue
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = 0;; ++u) {
            const int um = u % kMeta;
            if (!mbar_wait(mfull0 + 8u * um, (uint32_t)(u / kMeta) & 1u, kWaitNs)) {
                if (lane == 0) timeout(p);
                break;
            }
            const UnitMeta &m = meta[um];
            const int n = m.n;
            if (n < 0) break;
            if (n > 0) {
                if (!mbar_wait(tfull0 + 8u * acc, acc_phase, kWaitNs)) {
                    if (lane == 0) timeout(p);
                    break;
                }
                tc_fence_after();
                const int t = warp * kWarp + lane;
                const int tok = m.tok[t];
                const uint32_t trow = tmem_base + ((uint32_t)(warp * kWarp) << 16) + (uint32_t)(acc * kMaxN);
                for (int c0 = 0; c0 < m.npad; c0 += 16) {
                    uint32_t r[16];
                    tmem_load_16(trow + (uint32_t)c0, r);
                    tmem_wait_load();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = c0 + j;
                        if (col >= n) break;
                        const float v = __uint_as_float(r[j]);
                        const int row = m.rows[col];
                        if (SCATTER) {
                            if (tok >= 0) p.out_logits[(size_t)row * p.V + tok] = v;
                        } else {
                            unsigned long long key = tok >= 0 ? argmax_key(v, tok) : 0ull;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) {
                                const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
                                key = other > key ? other : key;
                            }
                            if (lane == 0 && key) atomicMax(best + row, key);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mempty0 + 8u * um);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
    if (SCATTER) return;
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
        const unsigned long long k = best[b];
        if (k) atomicMax(p.keys + b, k);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(p.ctrl + kCtrlTicket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
        const unsigned long long k = atomicAdd(p.keys + b, 0ull);
        int32_t tok;
        float v;
        decode_argmax_key(k, &tok, &v);
        p.out_tokens[b] = tok;
        if (p.out_max) p.out_max[b] = v;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// bf16 [rows, inner] with row stride `stride` elements, read in boxes of 64 x
// box_rows (box_rows = 1 for tile::gather4).
bool encode_rows(CUtensorMap *map, const void *base, long long inner, long long rows, long long stride,
                 int box_rows)
{
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t gather_tc_smem_bytes(int B, int stages)
{
    return 1024 + (size_t)stages * (kABytes + (size_t)kMaxN * kTileK * 2) + kMeta * sizeof(UnitMeta) +
           (size_t)B * 8 + (size_t)(2 * stages + 4 + 2 * kMeta) * 8 + 16;
}

cudaError_t launch_gather_tc(const GatherParams &g, bool scatter, cudaStream_t s)
{
    Params p{};
    p.ordering = g.ordering;
    p.offsets = g.offsets;
    p.rowmask = g.rowmask;
    p.items = g.items;
    p.items_cap = g.items_cap;
    p.ctrl = g.ctrl;
    p.keys = g.keys;
    p.out_logits = g.out_logits;
    p.out_tokens = g.out_tokens;
    p.out_max = g.out_max;
    p.B = g.B;
    p.H = g.H;
    p.V = g.V;
    p.S = g.S;
    p.W = g.W;
    p.C = g.C;
    p.chunk = g.chunk;
    if (p.chunk > kTileM) return cudaErrorInvalidValue;
    p.num_kb = (g.H + kTileK - 1) / kTileK;
    int stages = 6;
    while (stages > 2 && gather_tc_smem_bytes(g.B, stages) > 220 * 1024) --stages;
    p.stages = stages;
    alignas(64) CUtensorMap map_e;
    alignas(64) CUtensorMap map_h;
    p.ordered = g.embed_ordered != nullptr;
    if (p.ordered ? !encode_rows(&map_e, g.embed_ordered, g.H, g.V, g.ld, kTileM)
                  : !encode_rows(&map_e, g.embed, g.H, g.V, g.ld, 1))
        return cudaErrorInvalidValue;
    if (!encode_rows(&map_h, g.hidden, g.H, g.B, g.H, 1)) return cudaErrorInvalidValue;
    const size_t smem = gather_tc_smem_bytes(g.B, stages);
    if (scatter) {
        cudaError_t e = allow_smem((const void *)k_gather_tc<true>, smem);
        if (e != cudaSuccess) return e;
        return launch_dependent(k_gather_tc<true>, dim3(sm_count()), dim3(kThreads), smem, s, map_e, map_h, p);
    }
    cudaError_t e = allow_smem((const void *)k_gather_tc<false>, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_gather_tc<false>, dim3(sm_count()), dim3(kThreads), smem, s, map_e, map_h, p);
}

}  // namespace mtp
