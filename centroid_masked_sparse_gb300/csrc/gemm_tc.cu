// Tensor-core skinny GEMM for the centroid projection and the dense head:
//   out[n, m] = sum_k T[m, k] * h[n, k]      (T = centroid table or lm_head table)
//
// The centroid Linear of Gemma4MTPMaskedEmbedder._select_and_score and the
// dense LogitsProcessor head of Gemma4MTP.compute_logits ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py) are both
// a bf16 table times a small batch of hidden states.  Once the batch is a few
// rows the contraction is worth the tensor cores: the table is the MMA's M
// side (128 rows a tile, in the 128 TMEM lanes) and the batch is N (padded to
// a multiple of 16, at most 256), so every table byte is read from HBM once
// and the batch operand is reused out of shared memory.
//
// Six warps per CTA (the persistent dense head runs one CTA per SM):
//   warp 4  one thread issues TMA loads of 128x64 table tiles and Nx64 batch
//           tiles (128-byte swizzle) into a ring of shared-memory stages;
//   warp 5  one thread issues tcgen05.mma (kind::f16, fp32 accumulate) into a
//           double-buffered TMEM accumulator and commits stage releases;
//   warps 0-3 read the accumulator with tcgen05.ld (one row per thread) and
//           write fp32 results; for the dense head they also fold each row's
//           (logit, lower token id) argmax key into a 64-bit atomicMax.
// Split-K (for the projection, whose M is only C): the splits of one output
// tile run as one thread-block cluster; each CTA parks its partial tile in its
// own shared memory and rank 0 adds the partials through distributed shared
// memory in rank order, so results are deterministic and no partial ever goes
// to HBM.  Every mbarrier wait gives up after a wall-clock limit and records
// MTP_DEVERR_TIMEOUT instead of hanging.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace mtp {

using namespace sm100;

namespace {

constexpr int kTcThreads = 192;
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr uint32_t kABytes = kTileM * kTileK * 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr int kMaxStages = 8;

struct TcParams {
    int M, N, K;
    int n_pad, n_blocks, num_kb, splits, kb_per_split, m_tiles, units, stages;
    uint32_t tmem_cols;
    float *out;
    long long ldo, split_stride;
    unsigned long long *keys;
    uint32_t *ctrl;         // [0] error word, [2] ticket (argmax only)
    int32_t *out_tokens;
    float *out_max;
    uint32_t *err;          // timeout reports (may be null)
    uint32_t *zero;         // cleared at kernel start (the next kernels' workspace words)
    int zero_words;
    int cluster_reduce;     // splits > 1: one cluster per output tile, summed through DSMEM
    int round_bf16;         // dense head: logits rounded to bf16 before they are stored or compared
    float softcap;          // dense head: final logit softcap (cap * tanh(v / cap)), 0 = none
    int after_stage;        // launched behind the staging of the hidden rows: the producer
                            // waits for it (griddepcontrol.wait) before its first load
};

// Unit u = (m tile, n block, k split) with the split innermost, so that the
// splits of one output tile are consecutive CTAs: one thread-block cluster.
__device__ __forceinline__ void decode_unit(const TcParams &p, int u, int *mt, int *sp, int *nb)
{
    *sp = u % p.splits;
    u /= p.splits;
    *nb = u % p.n_blocks;
    *mt = u / p.n_blocks;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_addr, uint32_t rank)
{
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}

// Plain (non-volatile) distributed-shared-memory load, so independent loads overlap;
// the cluster barriers around the reduction order it against the writes.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr)
{
    float v;
    asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Columns of the partial tile that one reduction step loads at once (from every rank).
constexpr int kRedCols = 4;

__device__ __forceinline__ void report_timeout(const TcParams &p)
{
    if (p.err) atomicOr(p.err, MTP_DEVERR_TIMEOUT);
}

__global__ void __launch_bounds__(kTcThreads)
    k_tc_gemm(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
              const TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages;
    const uint32_t b_bytes = (uint32_t)p.n_pad * kTileK * 2;
    uint8_t *a_smem = smem;
    uint8_t *b_smem = smem + (size_t)S * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(b_smem + (size_t)S * b_bytes);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    __shared__ int s_last;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x & (kWarp - 1);
    // let the next kernel of the call (the top-K) be scheduled now; it waits for our results
    asm volatile("griddepcontrol.launch_dependents;");
    for (int i = blockIdx.x * kTcThreads + threadIdx.x; i < p.zero_words; i += gridDim.x * kTcThreads)
        p.zero[i] = 0u;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);
    const uint32_t tfull0 = smem_u32(bars + 2 * S);
    const uint32_t tempty0 = smem_u32(bars + 2 * S + 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, 4);
        }
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 4) {
        if (lane == 0) {
            tma_prefetch_map(&tmap_a);
            tma_prefetch_map(&tmap_b);
            // the B operand (hidden rows) is written by the staging kernel before this one
            if (p.after_stage) asm volatile("griddepcontrol.wait;" ::: "memory");
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int mt, sp, nb;
                decode_unit(p, u, &mt, &sp, &nb);
                const int kb0 = sp * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * stage, kABytes + b_bytes);
                    tma_load_2d(smem_u32(a_smem + (size_t)stage * kABytes), &tmap_a, kb * kTileK,
                                mt * kTileM, full0 + 8 * stage);
                    tma_load_2d(smem_u32(b_smem + (size_t)stage * b_bytes), &tmap_b, kb * kTileK,
                                nb * p.n_pad, full0 + 8 * stage);
                    armed |= 1u << stage;
                    armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                report_timeout(p);
                // let the copies already issued land before the CTA leaves
                for (int s = 0; s < S; ++s)
                    if (armed >> s & 1u) mbar_wait(full0 + 8 * s, armed_par >> s & 1u, 10000000ull);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kTileM, p.n_pad);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                int mt, sp, nb;
                decode_unit(p, u, &mt, &sp, &nb);
                const int kb0 = sp * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.n_pad);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full0 + 8 * stage, phase, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_kmajor_desc(smem_u32(a_smem + (size_t)stage * kABytes));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(b_smem + (size_t)stage * b_bytes));
#pragma unroll
                    for (int k = 0; k < kTileK / 16; ++k)
                        mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    mma_commit(empty0 + 8 * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) report_timeout(p);
        }
    } else {
        // epilogue: warp w owns TMEM lanes (tile rows) 32w .. 32w+31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            int mt, sp, nb;
            decode_unit(p, u, &mt, &sp, &nb);
            if (!mbar_wait(tfull0 + 8 * acc, acc_phase, kWaitLimitNs)) {
                if (lane == 0) report_timeout(p);
                break;
            }
            tc_fence_after();
            const int m = mt * kTileM + warp * kWarp + lane;
            const bool m_ok = m < p.M;
            const uint32_t trow = tmem_base + ((uint32_t)(warp * kWarp) << 16) + (uint32_t)(acc * p.n_pad);
            float *outp = p.out ? p.out + (size_t)sp * p.split_stride : nullptr;
            // cluster mode: the stage ring is idle now (every MMA of this CTA's only
            // unit has completed), so it holds the partial tile as red[n][128]: a warp
            // reads one column of it as one contiguous 128-byte line
            float *red = reinterpret_cast<float *>(smem);
            const int m_local = warp * kWarp + lane;
            for (int c0 = 0; c0 < p.n_pad; c0 += 16) {
                uint32_t r[16];
                tmem_load_16(trow + (uint32_t)c0, r);
                tmem_wait_load();
                if (p.cluster_reduce) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) red[(c0 + j) * kTileM + m_local] = __uint_as_float(r[j]);
                    continue;
                }
                // the dense head's options act on the 16 loaded values before any
                // store or comparison, behind one uniform test per group
                if (p.softcap > 0.f || p.round_bf16) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float v = __uint_as_float(r[j]);
                        if (p.softcap > 0.f) v = p.softcap * tanhf(v / p.softcap);
                        if (p.round_bf16) v = round_bf16(v);
                        r[j] = __float_as_uint(v);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = nb * p.n_pad + c0 + j;
                    if (n >= p.N) break;
                    const float v = __uint_as_float(r[j]);
                    if (outp && m_ok) outp[(size_t)n * p.ldo + m] = v;
                    if (p.keys) {
                        unsigned long long key = m_ok ? argmax_key(v, m) : 0ull;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
                            key = other > key ? other : key;
                        }
                        if (lane == 0 && key) atomicMax(p.keys + n, key);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    if (p.cluster_reduce) {
        // split-K: the cluster's CTAs hold the partial tiles of one output tile.  Each
        // rank sums a slice of the columns over all ranks, in rank order (deterministic),
        // and stores it; it loads kRedCols columns from every rank at once (all loads
        // independent, each warp-wide load one 128-byte line), so the remote latency is
        // paid once per group of columns, not once per column.
        cluster_sync_all();
        uint32_t rank;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        if (warp < 4) {
            int mt, sp, nb;
            decode_unit(p, blockIdx.x, &mt, &sp, &nb);
            const int m_local = warp * kWarp + lane;
            const int m = mt * kTileM + m_local;
            const int per = (p.n_pad + p.splits - 1) / p.splits;
            const int j0 = (int)rank * per, j1 = min(p.n_pad, j0 + per);
            const uint32_t red0 = smem_u32(smem);
            uint32_t base[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) base[r] = r < p.splits ? dsmem_addr(red0, (uint32_t)r) : 0u;
            if (m < p.M) {
                for (int j = j0; j < j1; j += kRedCols) {
                    float part[kRedCols][8];
#pragma unroll
                    for (int q = 0; q < kRedCols; ++q) {
                        const uint32_t off = (uint32_t)(((j + q) * kTileM + m_local) * 4);
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            part[q][r] = (r < p.splits && j + q < j1) ? ld_dsmem_f32(base[r] + off) : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < kRedCols; ++q) {
                        const int n = nb * p.n_pad + j + q;
                        if (j + q >= j1 || n >= p.N) break;
                        float v = 0.f;
#pragma unroll
                        for (int r = 0; r < 8; ++r) v += part[q][r];   // rank order: deterministic
                        p.out[(size_t)n * p.ldo + m] = v;
                    }
                }
            }
        }
        // no CTA leaves while another still reads its shared memory: a thread's loads have
        // returned their values (summed and stored) before it arrives, so the arrive needs
        // no release (a released arrive waits for the stores and measured ~0.5 us slower)
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    }
    // launched behind the scatter's fill (which it does not read): complete only after it,
    // so that every later kernel of the call sees the fill done (no-op otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!p.keys) return;
    // the last CTA to finish turns the argmax keys into token ids
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(p.ctrl + kCtrlTicket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int b = threadIdx.x; b < p.N; b += kTcThreads) {
        const unsigned long long k = atomicAdd(p.keys + b, 0ull);
        int32_t tok;
        float v;
        decode_argmax_key(k, &tok, &v);
        p.out_tokens[b] = tok;
        if (p.out_max) p.out_max[b] = v;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
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

// Row-major bf16 matrix [rows, inner] (row stride in elements) as 64 x box_rows tiles.
bool encode_map(CUtensorMap *map, const void *base, long long inner, long long rows,
                long long row_stride, int box_rows)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_stride * 2};
    cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int tc_n_pad(int N)
{
    const int n = N < 256 ? N : 256;
    return (n + 15) / 16 * 16;
}

int tc_splits(int M, int N, int K)
{
    // aim at ~128 CTAs streaming the table; at most 8 splits (a portable cluster)
    const int m_tiles = (M + kTileM - 1) / kTileM;
    const int n_blocks = (N + 255) / 256;
    const int num_kb = (K + kTileK - 1) / kTileK;
    int splits = 128 / (m_tiles * n_blocks);
    if (splits > 8) splits = 8;
    // long contractions keep longer splits: at K = 2560 (40 k-blocks), M = 2048, N = 64 four
    // splits of 10 k-blocks measured faster than eight of 5 (projection + top-K 19.4 vs
    // 25.3 us on GB300); at K = 1536 eight splits of 3 stay ahead (17.4 vs 18.2 us)
    if (num_kb >= 32 && splits > 4) splits = 4;
    if (splits > num_kb) splits = num_kb;
    if (splits < 1) splits = 1;
    const int per = (num_kb + splits - 1) / splits;  // no empty split
    return (num_kb + per - 1) / per;
}

cudaError_t launch_tc_gemm(const TcGemmArgs &a, cudaStream_t s)
{
    TcParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.n_pad = tc_n_pad(a.N);
    p.n_blocks = (a.N + p.n_pad - 1) / p.n_pad;
    p.num_kb = (a.K + kTileK - 1) / kTileK;
    p.splits = a.splits < 1 ? 1 : a.splits;
    p.kb_per_split = (p.num_kb + p.splits - 1) / p.splits;
    p.m_tiles = (a.M + kTileM - 1) / kTileM;
    p.units = p.m_tiles * p.splits * p.n_blocks;
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.n_pad)) cols <<= 1;
    p.tmem_cols = cols;
    const size_t stage_bytes = kABytes + (size_t)p.n_pad * kTileK * 2;
    const size_t budget = 220 * 1024 - 1024 - 256;
    int stages = (int)(budget / stage_bytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (p.splits > 1) {
        // one unit per CTA: enough stages for its k-blocks and for the partial tile that the
        // cluster reduction parks in the ring; less shared memory lets several CTAs share an
        // SM, so every cluster of the grid is resident at once
        const size_t red = (size_t)p.n_pad * kTileM * 4;
        int need = p.kb_per_split;
        while ((size_t)need * stage_bytes < red) ++need;
        if (need < 2) need = 2;
        if (need < stages) stages = need;
    }
    if (stages < 2) return cudaErrorInvalidValue;
    p.stages = stages;
    p.out = a.out;
    p.ldo = a.ldo;
    p.split_stride = 0;
    p.keys = a.keys;
    p.ctrl = a.ctrl;
    p.out_tokens = a.out_tokens;
    p.out_max = a.out_max;
    p.err = a.ctrl ? a.ctrl + kCtrlError : nullptr;
    p.zero = a.zero;
    p.zero_words = a.zero ? a.zero_words : 0;
    p.cluster_reduce = p.splits > 1;
    p.round_bf16 = a.round_bf16 ? 1 : 0;
    p.softcap = a.softcap;
    p.after_stage = a.after_stage ? 1 : 0;
    if (p.cluster_reduce && (size_t)stages * stage_bytes < (size_t)p.n_pad * kTileM * 4)
        return cudaErrorInvalidValue;
    if (p.cluster_reduce && (p.keys || p.splits > 8 || p.units > 65535)) return cudaErrorInvalidValue;

    alignas(64) CUtensorMap map_a;
    alignas(64) CUtensorMap map_b;
    if (!encode_map(&map_a, a.table, a.K, a.M, a.ld_table, kTileM)) return cudaErrorInvalidValue;
    if (!encode_map(&map_b, a.hidden, a.K, a.N, a.K, p.n_pad)) return cudaErrorInvalidValue;

    const size_t smem = 1024 + (size_t)stages * stage_bytes + (size_t)(2 * stages + 4) * 8 + 16;
    cudaError_t e = allow_smem((const void *)k_tc_gemm, smem);
    if (e != cudaSuccess) return e;
    if (!p.cluster_reduce) {
        int grid = sm_count();
        if (grid > p.units) grid = p.units;
        if (a.after_fill || a.after_stage)
            return launch_dependent(k_tc_gemm, dim3(grid), dim3(kTcThreads), smem, s, map_a, map_b, p);
        k_tc_gemm<<<grid, kTcThreads, smem, s>>>(map_a, map_b, p);
        return cudaGetLastError();
    }
    // one CTA per unit, the splits of a tile in one cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.units, 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (a.after_fill || a.after_stage) ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k_tc_gemm, map_a, map_b, p);
}

}  // namespace mtp
