// Host-side interface between the C ABI (mtp_head.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace mtp {

// Number of 256-element chunks a warp covers for rows of H bf16 values, rounded
// up to a compiled size; 0 if H is beyond the compiled sizes.
int chunks_for_hidden(int H);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Resident CTAs per SM for a kernel (cached per kernel and shared-memory size).
int blocks_per_sm(const void *kernel, int block, size_t smem);

// Raise a kernel's dynamic shared-memory limit to at least `smem` (cached per kernel
// and device; done for any nonzero size, since static shared memory shares the limit).
cudaError_t allow_smem(const void *kernel, size_t smem);

// Host-side argument checks of the sparse-argmax call (descriptor, batch, pointers,
// alignment), shared by its workspace and allocation-free entry points.
mtp_status check_topk_call(const mtp_head_desc *desc, const void *hidden, int32_t batch, const int32_t *out_tokens);

// Makes `dev` current for the rest of a call and gives the calling thread back its
// own current device when the call returns (ok == false: either step failed).
struct DeviceScope {
    int prev = -1;
    bool ok = false;
    explicit DeviceScope(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceScope()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;
};

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel on the stream is still running and must execute
// griddepcontrol.wait before it reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kProjThreads = 256;
constexpr int kProjRowsPerWarp = 2;
constexpr int kTopkThreads = 256;

cudaError_t launch_projection(const ProjParams &p, cudaStream_t s);
cudaError_t launch_topk(const TopkParams &p, cudaStream_t s);
// Gather-score kernel (score.cu): ring/row-group geometry, its shared memory, launch.
void gather_geometry(GatherParams &p);
size_t gather_smem_bytes(const GatherParams &p);
cudaError_t launch_gather(const GatherParams &p, bool scatter, cudaStream_t s);
// Direct CUDA-core variant for batches of at most 32 rows (score.cu; no sparse pair);
// its hidden rows, B x H bf16, must fit in shared memory.
cudaError_t launch_gather_direct(const GatherParams &p, bool scatter, cudaStream_t s);
// Tensor-core variant of the gather (gather_tc.cu); p.chunk <= 128, a multiple of 32
// when p.packed is set.
cudaError_t launch_gather_tc(const GatherParams &p, bool scatter, cudaStream_t s);
constexpr int kTcGatherChunk = 128;
// Expected rows per selected cluster (B*K/C) from which the tensor-core gather is used.
constexpr int kTcGatherMinReuse = 4;
// Fused top-K + gather + finish for small batches (select_gather.cu): every CTA
// selects its row's top-K from p.scores itself; no buckets or work items.  K at most
// kSelectGatherMaxK; no sparse pair.
cudaError_t launch_select_gather(const GatherParams &p, bool scatter, cudaStream_t s);
constexpr int kSelectGatherMaxK = 1024;
// Wall-clock limit of a bounded mbarrier wait in the pipelined gather (mtp_wait_test
// can change it for a test).
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
// CTAs per SM of the fused kernel: more rows in flight with three, except for a single
// row (its ticket's arrivals) and long rows (measured on GB300: H=1536 B=2, 4, 8 21.4,
// 26.2, 36.7 against 21.8, 27.2, 38.1 us per call with two; B=1 19.6 against 19.3;
// H=2560 B=8 53.6 against 52.9)
constexpr int kSelectGatherCtasPerSm = 2;
constexpr int kSelectGatherCtasPerSmShort = 3;   // batches of 2 or more rows, H <= 1536
cudaError_t launch_fill(float *out, size_t n, float value, cudaStream_t s);
// Copy `bytes` (a multiple of 16, both ends 16-byte aligned) from memory the device can
// read (pinned host memory included) to device memory with one kernel.
cudaError_t launch_stage_rows(void *dst, const void *src, size_t bytes, cudaStream_t s);
// The packed embedding table of the tensor-core gather (gather_tc.cu): byte size for
// the shapes (an upper bound with explicit offsets) and the kernels that fill it.
// n = clusters the table holds (a shard's [c0, c1), or all C).
size_t packed_table_bytes(int V, int H, int C, int n, bool explicit_offsets);
size_t packed_poff_offset(int V, int H, int C, int n, bool explicit_offsets);
cudaError_t launch_pack_embeddings(const uint16_t *embed, long long ld, const int32_t *ordering,
                                   const int32_t *offsets, int V, int H, int C, int c0, int c1, uint8_t *packed,
                                   uint32_t *ctrl, cudaStream_t s);
// Argmax keys (u64, workspace) -> signed-comparable int64 keys, and back to token ids.
cudaError_t launch_export_keys(const unsigned long long *keys, int B, int64_t *out, cudaStream_t s);
cudaError_t launch_decode_keys(const int64_t *keys, int B, int32_t *tokens, float *maxv, cudaStream_t s);

// Tensor-core skinny GEMM out[n, m] = sum_k table[m, k] * hidden[n, k] (gemm_tc.cu).
struct TcGemmArgs {
    const void *table;      // bf16 [M, K], row stride ld_table elements
    long long ld_table;
    int M;
    const void *hidden;     // bf16 [N, K] contiguous
    int N, K;
    int splits;             // split-K factor (> 1: reduced inside a thread-block cluster)
    float *out;             // fp32, out[n * ldo + m] (may be null with keys)
    long long ldo;
    unsigned long long *keys;  // per-row argmax keys (dense head) or null
    uint32_t *ctrl;         // workspace control words: ticket for keys, error word
    int32_t *out_tokens;    // with keys
    float *out_max;         // with keys, optional
    bool round_bf16;        // round each output to bf16 first (dense head option)
    bool after_fill;        // launched behind the scatter's fill, overlapping it
    bool after_stage;       // launched behind the staging of host-resident hidden rows
    float softcap;          // dense head: cap * tanh(v / cap) for cap > 0
    uint32_t *zero;         // words cleared at kernel start (may be null)
    int zero_words;
};
// The projection runs on tensor cores for batches above kCudaCoreProjBatch rows once
// B * H exceeds kCudaCoreProjMaxWork; otherwise the CUDA-core GEMV (whose per-row work
// grows with B * H while both read the table once, and which reduces up to eight rows
// at once) is ahead.  Measured on GB300 per call against the earlier rule (tensor cores
// from 4 rows once B * H > 8192): H=256 B=16 28.0 vs 30.9 us, B=32 31.9 vs 37.2, B=64
// 38.8 vs 41.5; H=1536 B=6 30.2 vs 31.8, B=8 34.1 vs 35.9; H=2560 B=4 33.5 vs 38.2, B=6
// 41.9 vs 45.1, B=8 49.3 vs 52.8.  Beyond the limit the GEMV lost: H=1536 B=12 45.3 vs
// 44.4, B=20 59.6 vs 57.8; H=2560 B=12 73.2 vs 66.4.
constexpr int kCudaCoreProjBatch = 8;
constexpr long long kCudaCoreProjMaxWork = 16384;
int tc_splits(int M, int N, int K);
cudaError_t launch_tc_gemm(const TcGemmArgs &a, cudaStream_t s);

}  // namespace mtp
