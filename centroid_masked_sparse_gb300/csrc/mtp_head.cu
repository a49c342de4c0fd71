// C ABI of the centroid-masked sparse LM head: argument checks, workspace
// layout and the launch sequence of each call.  Declarations and the contract
// of every entry point are in include/mtp_head.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "internal.h"

namespace mtp {

int chunks_for_hidden(int H)
{
    static const int sizes[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16};
    const int need = (H / 8 + kWarp - 1) / kWarp;
    for (int s : sizes)
        if (s >= need) return s;
    return 0;
}

static std::mutex g_cache_mu;

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    static std::unordered_map<int, int> cache;
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev] = n;
    return n;
}

struct FnKey {
    const void *fn;
    int dev;
    size_t smem;
    bool operator==(const FnKey &o) const { return fn == o.fn && dev == o.dev && smem == o.smem; }
};
struct FnKeyHash {
    size_t operator()(const FnKey &k) const
    {
        return std::hash<const void *>()(k.fn) ^ (std::hash<size_t>()(k.smem) * 31u) ^ (size_t)k.dev;
    }
};

int blocks_per_sm(const void *kernel, int block, size_t smem)
{
    int dev = 0;
    cudaGetDevice(&dev);
    static std::unordered_map<FnKey, int, FnKeyHash> cache;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        auto it = cache.find(FnKey{kernel, dev, smem});
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess) n = 1;
    std::lock_guard<std::mutex> lk(g_cache_mu);
    cache[FnKey{kernel, dev, smem}] = n;
    return n;
}

cudaError_t allow_smem(const void *kernel, size_t smem)
{
    // raised even below the default 48 KB: the kernel's static shared memory counts
    // against the same limit, so a dynamic size just under it can still fail to launch
    if (smem == 0) return cudaSuccess;
    int dev = 0;
    cudaGetDevice(&dev);
    static std::unordered_map<FnKey, size_t, FnKeyHash> done;  // keyed by (fn, dev)
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        auto it = done.find(FnKey{kernel, dev, 0});
        if (it != done.end() && it->second >= smem) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_cache_mu);
    done[FnKey{kernel, dev, 0}] = smem;
    return cudaSuccess;
}

}  // namespace mtp

using namespace mtp;

namespace {

constexpr int kMinChunk = 8;     // smallest work item (ordered positions); sizes the item list
constexpr int kMaxChunk = 64;

void *g_prof[5][2] = {};

struct Layout {
    size_t ctrl, keys, ccount, rowmask, zero_end, scores, topk, items, hidden, total;
    int W;
    int items_cap;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

Layout layout_for(const mtp_head_desc *d, int B)
{
    Layout L{};
    const size_t C = (size_t)d->num_centroids, K = (size_t)d->top_k, V = (size_t)d->vocab_size;
    L.W = (B + 31) / 32;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.ctrl = take(kCtrlWords * sizeof(uint32_t));
    L.keys = take((size_t)B * sizeof(unsigned long long));
    L.ccount = take(C * sizeof(int32_t));
    L.rowmask = take(C * (size_t)L.W * sizeof(uint32_t));
    L.zero_end = off;
    L.scores = take((size_t)B * C * sizeof(float));
    L.topk = take((size_t)B * K * sizeof(int32_t));
    const size_t nsel = C < (size_t)B * K ? C : (size_t)B * K;
    const size_t max_items = V / kMinChunk + nsel + 1;
    L.items = take(max_items * sizeof(int2));
    L.items_cap = (int)max_items;
    // the staged copy of host-resident hidden states (last, so that a call with fewer
    // rows than the workspace was sized for still fits)
    L.hidden = (d->flags & MTP_FLAG_HOST_HIDDEN) ? take((size_t)B * d->hidden_size * 2) : off;
    L.total = off;
    return L;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// The clusters a descriptor owns: [cluster_begin, cluster_end), or all C for (0, 0).
void cluster_span(const mtp_head_desc *d, int *c0, int *c1)
{
    if (d->cluster_begin == 0 && d->cluster_end == 0) {
        *c0 = 0;
        *c1 = d->num_centroids;
    } else {
        *c0 = d->cluster_begin;
        *c1 = d->cluster_end;
    }
}

bool span_ok(const mtp_head_desc *d)
{
    if (d->cluster_begin == 0 && d->cluster_end == 0) return true;
    return d->cluster_begin >= 0 && d->cluster_begin <= d->cluster_end && d->cluster_end <= d->num_centroids;
}

// Checks of the descriptor.  `centroids`: the call reads the centroid table
// (and needs C, K); `embed`: it reads the embedding table; `ordering`: it
// reads token_ordering.
mtp_status check_desc(const mtp_head_desc *d, bool centroids, bool embed, bool ordering)
{
    if (!d) return MTP_ERR_NULL;
    if ((embed && !d->embed_w) || (centroids && !d->centroid_w) || (ordering && !d->token_ordering))
        return MTP_ERR_NULL;
    if (d->vocab_size < 1 || d->hidden_size < 8 || d->hidden_size % 8 != 0) return MTP_ERR_SHAPE;
    if (d->hidden_size > MTP_MAX_HIDDEN) return MTP_ERR_UNSUPPORTED;
    if (d->device < 0) return MTP_ERR_SHAPE;
    if (embed) {
        if (d->ld_embed < d->hidden_size) return MTP_ERR_SHAPE;
        if (d->ld_embed % 8 != 0 || !aligned16(d->embed_w)) return MTP_ERR_ALIGN;
        if (((uintptr_t)d->embed_packed & 255u) != 0) return MTP_ERR_ALIGN;
    }
    if (centroids) {
        if (d->num_centroids < 1 || d->top_k < 1 || d->top_k > d->num_centroids) return MTP_ERR_SHAPE;
        if (d->num_centroids > MTP_MAX_CENTROIDS) return MTP_ERR_UNSUPPORTED;
        if (!aligned16(d->centroid_w)) return MTP_ERR_ALIGN;
        if (!span_ok(d)) return MTP_ERR_SHAPE;
    }
    if (d->flags & ~(MTP_FLAG_FILL_FINFO_MIN | MTP_FLAG_BF16_SCORES | MTP_FLAG_BF16_LOGITS | MTP_FLAG_HOST_HIDDEN))
        return MTP_ERR_UNSUPPORTED;
    if (!(d->final_logit_softcap >= 0.f)) return MTP_ERR_SHAPE;   // negative or NaN
    if (ordering && !d->cluster_offsets && (d->num_centroids < 1 || d->vocab_size % d->num_centroids != 0))
        return MTP_ERR_SHAPE;
    return MTP_OK;
}

mtp_status check_batch(int32_t B)
{
    if (B < 0) return MTP_ERR_SHAPE;
    if (B > MTP_MAX_BATCH) return MTP_ERR_UNSUPPORTED;
    return MTP_OK;
}

int proj_rows_per_group(int B, int H)
{
    int r = 49152 / (2 * H);
    if (r < 1) r = 1;
    return r < B ? r : B;
}

struct Prof {
    int id;
    cudaStream_t s;
    bool on;
    Prof(int id_, cudaStream_t s_) : id(id_), s(s_), on(false)
    {
        if (!g_prof[id][0] && !g_prof[id][1]) return;
        // never record the profiling events into a graph being captured
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        on = cudaStreamIsCapturing(s, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone;
        if (on && g_prof[id][0]) cudaEventRecord((cudaEvent_t)g_prof[id][0], s);
    }
    ~Prof()
    {
        if (on && g_prof[id][1]) cudaEventRecord((cudaEvent_t)g_prof[id][1], s);
    }
};

mtp_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA; }

// MTP_FLAG_HOST_HIDDEN: check that the device can read `hidden` (pinned or registered
// host memory at its device address, managed memory, or this GPU's memory), copy the
// batch's rows into the workspace's staging region with one kernel, and point the
// rest of the call at that copy.  Launches nothing when the pointer is unusable.
mtp_status stage_hidden(const mtp_head_desc *d, const void **hidden, int B, char *ws, const Layout &L,
                        cudaStream_t s)
{
    if (!(d->flags & MTP_FLAG_HOST_HIDDEN)) return MTP_OK;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, *hidden) != cudaSuccess) {
        cudaGetLastError();   // the failed query also sets the runtime's last error
        return MTP_ERR_UNSUPPORTED;
    }
    if (a.type == cudaMemoryTypeUnregistered || a.devicePointer != *hidden) return MTP_ERR_UNSUPPORTED;
    if (a.type == cudaMemoryTypeDevice && a.device != d->device) return MTP_ERR_UNSUPPORTED;
    void *dst = ws + L.hidden;
    mtp_status st = cuda_status(launch_stage_rows(dst, *hidden, (size_t)B * d->hidden_size * 2, s));
    if (st != MTP_OK) return st;
    *hidden = dst;
    return MTP_OK;
}

// Steps 1-2: projection (+ workspace reset) and top-K (+ bucketing when rowmask is set).
mtp_status run_select(const mtp_head_desc *d, const void *hidden, int B, float *scores,
                      int32_t *topk, char *ws, const Layout *L, int chunk, cudaStream_t s,
                      bool after_fill = false, bool after_stage = false)
{
    if (B > kCudaCoreProjBatch && (long long)B * d->hidden_size > kCudaCoreProjMaxWork) {
        // tensor cores: M = C centroid rows, N = batch, K = H, split-K in a cluster
        TcGemmArgs g{};
        g.table = d->centroid_w;
        g.ld_table = d->hidden_size;
        g.M = d->num_centroids;
        g.hidden = hidden;
        g.N = B;
        g.K = d->hidden_size;
        g.splits = tc_splits(g.M, g.N, g.K);
        g.out = scores;
        g.ldo = d->num_centroids;
        g.ctrl = ws ? (uint32_t *)ws : nullptr;
        g.zero = ws ? (uint32_t *)ws : nullptr;
        g.zero_words = ws ? (int)(L->zero_end / sizeof(uint32_t)) : 0;
        g.after_fill = after_fill;
        g.after_stage = after_stage;
        Prof pr(MTP_KERNEL_PROJECTION, s);
        mtp_status st = cuda_status(launch_tc_gemm(g, s));
        if (st != MTP_OK) return st;
    } else {
        ProjParams pp{};
        pp.hidden = (const uint16_t *)hidden;
        pp.wc = (const uint16_t *)d->centroid_w;
        pp.scores = scores;
        pp.zero = ws ? (uint32_t *)ws : nullptr;
        pp.zero_words = ws ? (int)(L->zero_end / sizeof(uint32_t)) : 0;
        pp.B = B;
        pp.H = d->hidden_size;
        pp.C = d->num_centroids;
        pp.rows_per_group = proj_rows_per_group(B, d->hidden_size);
        pp.after_fill = after_fill ? 1 : 0;
        pp.after_stage = after_stage ? 1 : 0;
        Prof pr(MTP_KERNEL_PROJECTION, s);
        mtp_status st = cuda_status(launch_projection(pp, s));
        if (st != MTP_OK) return st;
    }
    if (!topk) return MTP_OK;
    TopkParams tp{};
    tp.bf16_scores = (d->flags & MTP_FLAG_BF16_SCORES) ? 1 : 0;
    tp.scores = scores;
    tp.topk = topk;
    tp.B = B;
    tp.C = d->num_centroids;
    tp.K = d->top_k;
    tp.V = d->vocab_size;
    tp.S = d->cluster_offsets ? 0 : d->vocab_size / d->num_centroids;
    tp.offsets = d->cluster_offsets;
    if (ws) {
        tp.rowmask = (uint32_t *)(ws + L->rowmask);
        tp.W = L->W;
        tp.ccount = (int32_t *)(ws + L->ccount);
        tp.items = (int2 *)(ws + L->items);
        tp.items_cap = L->items_cap;
        tp.ctrl = (uint32_t *)ws;
        tp.chunk = chunk;
        cluster_span(d, &tp.c_begin, &tp.c_end);
    }
    Prof pr(MTP_KERNEL_TOPK, s);
    return cuda_status(launch_topk(tp, s));
}

// Positions per work item.  Small batches: few positions in all, so each gather
// CTA should get about one item (a CTA's producer walks its items one after the
// other, each paying a few dependent global loads); large batches: up to 64
// positions, which still leaves ~16 items per SM for the dynamic hand-out.
int choose_chunk(const mtp_head_desc *d, int B)
{
    const double avg = (double)d->vocab_size / d->num_centroids;
    const double est = (double)B * d->top_k * avg;
    const double per_cta = est / sm_count();
    int ch = kMinChunk;
    while (ch < kMaxChunk && ch < per_cta) ch *= 2;
    return ch;
}

// Hidden sizes whose 512-byte (or smaller) rows make per-row costs weigh most.
constexpr int kSmallHidden = 256;

// Which gather a call runs.  The tensor-core gather takes calls whose buckets are
// large (B*K >= 4C), where one candidate tile serves a whole bucket, and at
// H <= 256 calls from B*K >= C/4 on the token-order table too (its gathered tiles
// against the CUDA-core gather's row copies, measured on GB300 at H=256: B=64 52.3
// vs 93.9 us, B=16 33.2 vs 47.4 us; at H=1536 the CUDA-core gather stays ahead).
// With the packed embedding table it also takes calls with fewer (row, cluster) pairs: its
// block copies stream HBM faster than the CUDA-core gather's row copies and read
// no padding rows.  Running two or three CTAs per SM, it is ahead (measured on
// GB300) from B*K >= C/5 with uniform clusters (K=32, C=2048, H=1536: B=13, 14 48.4,
// 50.1 against 49.2, 52.7 us with the pipelined CUDA-core gather), from B*K >= C/4 with
// ragged ones (H=2560: B=13, 14 75.2, 75.9 against 72.6, 75.3 us, B=15 77.1 against
// 78.0; behind at C/8) and from B*K >= C/16 at H = 256, where the CUDA-core gather's
// per-row costs weigh most (behind at C/64).  Smaller calls keep more
// SMs busy with the CUDA-core gather's finer work items.  Its chunk is the largest
// of 128, 64, 32 positions that still gives about two work items per SM.
bool tc_gather_plan(const mtp_head_desc *d, int B, int *chunk)
{
    const long long pairs = (long long)B * d->top_k;
    const long long C = d->num_centroids;
    const bool large = pairs >= (long long)kTcGatherMinReuse * C;
    const bool packed_reuse =
        d->embed_packed && ((d->cluster_offsets ? 4 : 5) * pairs >= C ||
                            (d->hidden_size <= kSmallHidden && 16 * pairs >= C));
    if (d->embed_packed && (large || packed_reuse)) {
        const double avg = (double)d->vocab_size / d->num_centroids;
        const double clusters = (double)std::min<long long>(pairs, d->num_centroids);
        int ch = kTcGatherChunk;
        while (ch > 32 && clusters * (double)((long long)(avg + ch - 1) / ch) < 2.0 * sm_count()) ch /= 2;
        *chunk = ch;
        return true;
    }
    if (large || (d->hidden_size <= kSmallHidden && 4 * pairs >= C)) {
        *chunk = kTcGatherChunk;
        return true;
    }
    *chunk = choose_chunk(d, B);
    return false;
}

enum GatherKind { kGatherNone = -1, kGatherPipelined = 0, kGatherTensorCore = 1, kGatherDirect = 2, kGatherFused = 3 };

// Testing and profiling controls (mtp_force_gather, mtp_wait_test): process-wide.
std::atomic<int> g_force_kind{-1};
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall_test{0};

// Batches that run the fused top-K + gather kernel (select_gather.cu) behind the
// projection instead of the top-K kernel and a gather, for hidden sizes above
// kSmallHidden; at or below it the same batches take the direct gather.  With uniform
// clusters and H <= 1536 the fused kernel also takes 9 and 10 rows (measured on GB300
// against the direct gather: B=9 38.2 vs 40.1 us, B=10 40.2 vs 41.6; B=11 43.4 vs 42.5;
// ragged clusters at H=2560, B=9 and 10: 58.3 vs 54.4 and 61.5 vs 57.7).
constexpr int kFusedMaxBatch = 8;
constexpr int kFusedMaxBatchUniform = 10;
// The direct gather's batches at H <= kSmallHidden: up to 10 rows with the packed table
// (measured on GB300 against the tensor-core gather: B=9 24.1 vs 26.5 us, B=10 25.5 vs
// 25.8; B=12 level, B=14 27.7 vs 27.2), up to 20 on the token-order table (against the
// pipelined gather B=13, 15 27.4, 28.2 vs 40.3, 41.6 us; against the tensor-core one B=16,
// 20 29.4, 33.2 vs 32.4, 34.4; B=24 35.3 vs 34.9, B=32 40.7 vs 36.5).
constexpr int kDirectMaxBatchSmallHidden = 10;
constexpr int kDirectMaxBatchSmallHiddenTokenOrder = 20;

int fused_max_batch(const mtp_head_desc *d)
{
    return !d->cluster_offsets && d->hidden_size <= 1536 ? kFusedMaxBatchUniform : kFusedMaxBatch;
}

// Whether a gather kernel can run a masked call of this shape.
bool gather_can_run(const mtp_head_desc *d, int B, bool sparse, GatherKind k)
{
    switch (k) {
    case kGatherPipelined:
    case kGatherTensorCore: return true;
    case kGatherDirect: return !sparse && B <= 32 && (size_t)B * d->hidden_size * 2 <= 200u * 1024u;
    case kGatherFused: return !sparse && d->top_k <= kSelectGatherMaxK;
    default: return false;
    }
}

// The gather a masked call runs.  Batches of at most fused_max_batch rows at H > 256 take
// the fused kernel, which selects each row's top-K in the gather CTAs themselves.  The
// direct CUDA-core gather (each warp loads candidate rows straight into registers; no
// producer, ring or hand-off, so its latency chain is short) takes the small batches at
// H <= 256 (up to the limits above), whose 512-byte rows make the fused kernel's row
// stream (every row's candidates, no dedup) the slower one, and up to 12 rows elsewhere
// where the tensor-core gather would not run.  Measured on GB300 against the
// alternatives: uniform clusters B=12 ~46 vs ~47.5 us (pipelined), B=16 ~56.5 vs ~54.5 us
// (tensor cores); H=256 with the packed table, direct against fused (and tensor cores):
// B=1 18.1 vs 19.2, B=2 18.3 vs 19.9, B=4 21.1 vs 20.4, B=6 22.8 vs 26.6 (24.4), B=8 24.7
// vs 26.9 (26.9) us.  The sparse pair keeps the pipelined and tensor-core gathers.  A
// kind forced by mtp_force_gather that cannot run the call gives kGatherNone.
GatherKind gather_kind(const mtp_head_desc *d, int B, bool sparse, int *chunk)
{
    int tc_chunk = 0;
    const bool tc = tc_gather_plan(d, B, &tc_chunk);
    const int forced = g_force_kind.load(std::memory_order_relaxed);
    GatherKind k;
    if (forced >= 0) {
        k = (GatherKind)forced;
        if (!gather_can_run(d, B, sparse, k)) return kGatherNone;
    } else if (!sparse && B <= fused_max_batch(d) && d->hidden_size > kSmallHidden &&
               gather_can_run(d, B, sparse, kGatherFused)) {
        k = kGatherFused;
    } else if (!sparse &&
               B <= (d->hidden_size > kSmallHidden ? kFusedMaxBatch
                     : d->embed_packed             ? kDirectMaxBatchSmallHidden
                                                   : kDirectMaxBatchSmallHiddenTokenOrder) &&
               gather_can_run(d, B, sparse, kGatherDirect)) {
        k = kGatherDirect;
    } else if (!sparse && !tc && B <= 12) {
        k = kGatherDirect;
    } else {
        k = tc ? kGatherTensorCore : kGatherPipelined;
    }
    *chunk = k == kGatherTensorCore ? (tc ? tc_chunk : kTcGatherChunk) : choose_chunk(d, B);
    return k;
}

// The masked calls.  Finishes: the sparse argmax (out_tokens), the full-vocabulary
// scatter (out_logits [B, V]) or, with `sparse`, the sparse pair (out_logits and
// out_ids [B, K*S], every entry written, so no -inf fill).
mtp_status run_masked(const mtp_head_desc *d, const void *hidden, int B, int32_t *out_tokens,
                      float *out_max, float *out_logits, int32_t *out_ids, bool sparse, void *workspace,
                      size_t ws_bytes, cudaStream_t s)
{
    const Layout L = layout_for(d, B);
    if (!workspace || ws_bytes < L.total) return MTP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MTP_ERR_ALIGN;
    int chunk = 0;
    const GatherKind kind = gather_kind(d, B, sparse, &chunk);
    if (kind == kGatherNone) return MTP_ERR_UNSUPPORTED;
    const DeviceScope dev(d->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    mtp_status st = MTP_OK;
    char *ws = (char *)workspace;
    if ((st = stage_hidden(d, &hidden, B, ws, L, s)) != MTP_OK) return st;
    if (out_logits && !sparse) {
        Prof pr(MTP_KERNEL_FILL, s);
        const float fill = (d->flags & MTP_FLAG_FILL_FINFO_MIN) ? -3.3895313892515355e38f : -INFINITY;
        st = cuda_status(launch_fill(out_logits, (size_t)B * d->vocab_size, fill, s));
        if (st != MTP_OK) return st;
    }
    const bool tc_gather = kind == kGatherTensorCore;
    const bool fused = kind == kGatherFused;
    // the projection starts behind the staging kernel (programmatic launch) when it is the
    // next kernel; behind the scatter's fill it is ordered by the fill's own launch.  The
    // fused kernel selects the top-K itself, so only the projection runs here then.
    const bool fill = out_logits && !sparse;
    st = run_select(d, hidden, B, (float *)(ws + L.scores), fused ? nullptr : (int32_t *)(ws + L.topk), ws, &L,
                    chunk, s, fill, (d->flags & MTP_FLAG_HOST_HIDDEN) && !fill);
    if (st != MTP_OK) return st;

    GatherParams gp{};
    gp.hidden = (const uint16_t *)hidden;
    gp.embed = (const uint16_t *)d->embed_w;
    gp.packed = tc_gather ? (const uint8_t *)d->embed_packed : nullptr;
    {
        int c0, c1;
        cluster_span(d, &c0, &c1);
        gp.packed_clusters = c1 - c0;
    }
    gp.ld = d->ld_embed;
    gp.ordering = d->token_ordering;
    gp.offsets = d->cluster_offsets;
    gp.rowmask = (const uint32_t *)(ws + L.rowmask);
    gp.items = (const int2 *)(ws + L.items);
    gp.items_cap = L.items_cap;
    gp.ctrl = (uint32_t *)ws;
    gp.keys = out_tokens ? (unsigned long long *)(ws + L.keys) : nullptr;
    gp.out_logits = out_logits;
    gp.out_tokens = out_tokens;
    gp.out_max = out_max;
    gp.topk = (const int32_t *)(ws + L.topk);
    gp.bf16_logits = (d->flags & MTP_FLAG_BF16_LOGITS) ? 1 : 0;
    gp.K = d->top_k;
    gp.sparse_width = sparse ? d->top_k * (d->vocab_size / d->num_centroids) : 0;
    gp.out_ids = sparse ? out_ids : nullptr;
    gp.B = B;
    gp.H = d->hidden_size;
    gp.V = d->vocab_size;
    gp.S = d->cluster_offsets ? 0 : d->vocab_size / d->num_centroids;
    gp.W = L.W;
    gp.C = d->num_centroids;
    gp.chunk = chunk;
    gp.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    gp.stall_test = g_stall_test.load(std::memory_order_relaxed);
    gp.scores = (const float *)(ws + L.scores);
    gp.bf16_scores = (d->flags & MTP_FLAG_BF16_SCORES) ? 1 : 0;
    cluster_span(d, &gp.c_begin, &gp.c_end);
    Prof pr(MTP_KERNEL_GATHER_SCORE, s);
    if (fused) return cuda_status(launch_select_gather(gp, out_logits != nullptr, s));
    if (tc_gather) return cuda_status(launch_gather_tc(gp, out_logits != nullptr, s));
    if (kind == kGatherDirect) return cuda_status(launch_gather_direct(gp, out_logits != nullptr, s));
    gather_geometry(gp);
    return cuda_status(launch_gather(gp, out_logits != nullptr, s));
}

}  // namespace

namespace mtp {

mtp_status check_topk_call(const mtp_head_desc *desc, const void *hidden, int32_t batch, const int32_t *out_tokens)
{
    mtp_status st = check_desc(desc, true, true, true);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (!hidden || !out_tokens) return MTP_ERR_NULL;
    if (!aligned16(hidden)) return MTP_ERR_ALIGN;
    return MTP_OK;
}

}  // namespace mtp

extern "C" {

size_t mtp_workspace_bytes(const mtp_head_desc *desc, int32_t max_batch)
{
    if (!desc || max_batch < 1 || max_batch > MTP_MAX_BATCH) return 0;
    if (desc->vocab_size < 1 || desc->num_centroids < 1 || desc->top_k < 1 ||
        desc->top_k > desc->num_centroids || desc->num_centroids > MTP_MAX_CENTROIDS)
        return 0;
    return layout_for(desc, max_batch).total;
}

mtp_status mtp_centroid_scores(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                               float *scores, int32_t *topk_idx, void *stream)
{
    mtp_status st = check_desc(desc, true, false, false);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (desc->flags & MTP_FLAG_HOST_HIDDEN) return MTP_ERR_UNSUPPORTED;   // no workspace to stage into
    if (!hidden || !scores) return MTP_ERR_NULL;
    if (!aligned16(hidden)) return MTP_ERR_ALIGN;
    const DeviceScope dev(desc->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    return run_select(desc, hidden, batch, scores, topk_idx, nullptr, nullptr, kMinChunk,
                      (cudaStream_t)stream);
}

mtp_status mtp_masked_topk_tokens(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                                  int32_t *out_tokens, float *out_max, void *workspace,
                                  size_t workspace_bytes, void *stream)
{
    const mtp_status st = mtp::check_topk_call(desc, hidden, batch, out_tokens);
    if (st != MTP_OK || batch == 0) return st;
    return run_masked(desc, hidden, batch, out_tokens, out_max, nullptr, nullptr, false, workspace, workspace_bytes,
                      (cudaStream_t)stream);
}

mtp_status mtp_masked_scatter_logits(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                                     float *out_logits, void *workspace, size_t workspace_bytes,
                                     void *stream)
{
    mtp_status st = check_desc(desc, true, true, true);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (!hidden || !out_logits) return MTP_ERR_NULL;
    if (!aligned16(hidden) || !aligned16(out_logits)) return MTP_ERR_ALIGN;
    return run_masked(desc, hidden, batch, nullptr, nullptr, out_logits, nullptr, false, workspace, workspace_bytes,
                      (cudaStream_t)stream);
}

mtp_status mtp_select_and_score(const mtp_head_desc *desc, const void *hidden, int32_t batch, float *out_logits,
                                int32_t *out_ids, void *workspace, size_t workspace_bytes, void *stream)
{
    mtp_status st = check_desc(desc, true, true, true);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (desc->cluster_offsets) return MTP_ERR_UNSUPPORTED;   // the pair's width K*S needs uniform clusters
    if (batch == 0) return MTP_OK;
    if (!hidden || !out_logits) return MTP_ERR_NULL;
    if (!aligned16(hidden)) return MTP_ERR_ALIGN;
    return run_masked(desc, hidden, batch, nullptr, nullptr, out_logits, out_ids, true, workspace, workspace_bytes,
                      (cudaStream_t)stream);
}

mtp_status mtp_dense_lm_head(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                             float *out_logits, int32_t *out_tokens, float *out_max,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    mtp_status st = check_desc(desc, false, true, false);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (!hidden || (!out_logits && !out_tokens)) return MTP_ERR_NULL;
    if (out_max && !out_tokens) return MTP_ERR_NULL;
    if (!aligned16(hidden)) return MTP_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    const bool host_hidden = (desc->flags & MTP_FLAG_HOST_HIDDEN) != 0;
    Layout L{};
    if (out_tokens || host_hidden) {
        // the workspace layout only depends on V, C, K, B (and the flags); C and K may be
        // unset for a dense head
        mtp_head_desc d = *desc;
        if (d.num_centroids < 1) d.num_centroids = 1;
        if (d.top_k < 1 || d.top_k > d.num_centroids) d.top_k = 1;
        L = layout_for(&d, batch);
        size_t need = out_tokens ? L.keys + (size_t)batch * sizeof(unsigned long long) : 0;
        if (host_hidden) need = std::max(need, L.hidden + (size_t)batch * desc->hidden_size * 2);
        if (!ws || workspace_bytes < need) return MTP_ERR_WORKSPACE;
        if (!aligned16(ws)) return MTP_ERR_ALIGN;
    }
    const DeviceScope dev(desc->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    if (out_tokens) {
        st = cuda_status(cudaMemsetAsync(ws, 0, L.keys + (size_t)batch * sizeof(unsigned long long), s));
        if (st != MTP_OK) return st;
    }
    // after the clear, so that the GEMM's programmatic launch follows the staging kernel
    if ((st = stage_hidden(desc, &hidden, batch, ws, L, s)) != MTP_OK) return st;
    TcGemmArgs g{};
    g.table = desc->embed_w;
    g.ld_table = desc->ld_embed;
    g.M = desc->vocab_size;
    g.hidden = hidden;
    g.N = batch;
    g.K = desc->hidden_size;
    g.splits = 1;
    g.out = out_logits;
    g.round_bf16 = (desc->flags & MTP_FLAG_BF16_LOGITS) != 0;
    g.softcap = desc->final_logit_softcap;
    g.ldo = desc->vocab_size;
    g.keys = out_tokens ? (unsigned long long *)(ws + L.keys) : nullptr;
    g.ctrl = out_tokens ? (uint32_t *)ws : nullptr;
    g.out_tokens = out_tokens;
    g.out_max = out_max;
    g.after_stage = host_hidden;
    Prof pr(MTP_KERNEL_DENSE, s);
    return cuda_status(launch_tc_gemm(g, s));
}

size_t mtp_packed_embeddings_bytes(const mtp_head_desc *desc)
{
    if (check_desc(desc, false, true, false) != MTP_OK) return 0;
    if (desc->num_centroids < 1 || desc->num_centroids > MTP_MAX_CENTROIDS) return 0;
    if (!desc->cluster_offsets && desc->vocab_size % desc->num_centroids != 0) return 0;
    if (!span_ok(desc)) return 0;
    int c0, c1;
    cluster_span(desc, &c0, &c1);
    return packed_table_bytes(desc->vocab_size, desc->hidden_size, desc->num_centroids, c1 - c0,
                              desc->cluster_offsets != nullptr);
}

mtp_status mtp_pack_embeddings(const mtp_head_desc *desc, void *packed, size_t packed_bytes, void *workspace,
                               void *stream)
{
    mtp_status st = check_desc(desc, false, true, false);
    if (st != MTP_OK) return st;
    if (!desc->token_ordering || !packed) return MTP_ERR_NULL;
    if (desc->num_centroids < 1) return MTP_ERR_SHAPE;
    if (desc->num_centroids > MTP_MAX_CENTROIDS) return MTP_ERR_UNSUPPORTED;
    if (!desc->cluster_offsets && desc->vocab_size % desc->num_centroids != 0) return MTP_ERR_SHAPE;
    if (!span_ok(desc)) return MTP_ERR_SHAPE;
    if (((uintptr_t)packed & 255u) != 0 || !aligned16(workspace)) return MTP_ERR_ALIGN;
    int c0, c1;
    cluster_span(desc, &c0, &c1);
    const size_t need = packed_table_bytes(desc->vocab_size, desc->hidden_size, desc->num_centroids, c1 - c0,
                                           desc->cluster_offsets != nullptr);
    if (packed_bytes < need) return MTP_ERR_WORKSPACE;
    const char *src = (const char *)desc->embed_w, *dst = (const char *)packed;
    const size_t src_bytes = (size_t)desc->vocab_size * desc->ld_embed * 2;
    if (src < dst + need && dst < src + src_bytes) return MTP_ERR_SHAPE;   // overlapping tables
    const DeviceScope dev(desc->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    return cuda_status(launch_pack_embeddings((const uint16_t *)desc->embed_w, desc->ld_embed,
                                              desc->token_ordering, desc->cluster_offsets, desc->vocab_size,
                                              desc->hidden_size, desc->num_centroids, c0, c1, (uint8_t *)packed,
                                              (uint32_t *)workspace, (cudaStream_t)stream));
}

mtp_status mtp_masked_topk_keys(const mtp_head_desc *desc, const void *hidden, int32_t batch, int64_t *out_keys,
                                void *workspace, size_t workspace_bytes, void *stream)
{
    mtp_status st = check_desc(desc, true, true, true);
    if (st != MTP_OK) return st;
    if ((st = check_batch(batch)) != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (!hidden || !out_keys) return MTP_ERR_NULL;
    if (!aligned16(hidden)) return MTP_ERR_ALIGN;
    if (!workspace || workspace_bytes < layout_for(desc, batch).total) return MTP_ERR_WORKSPACE;
    // the call's decoded tokens go to the scores region, which nothing reads after the
    // top-K; the keys it leaves in the workspace are exported
    const Layout L = layout_for(desc, batch);
    const DeviceScope dev(desc->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    char *ws = (char *)workspace;
    st = run_masked(desc, hidden, batch, (int32_t *)(ws + L.scores), nullptr, nullptr, nullptr, false, workspace,
                    workspace_bytes, (cudaStream_t)stream);
    if (st != MTP_OK) return st;
    return cuda_status(launch_export_keys((const unsigned long long *)(ws + L.keys), batch, out_keys,
                                          (cudaStream_t)stream));
}

mtp_status mtp_decode_keys(const int64_t *keys, int32_t batch, int32_t *out_tokens, float *out_max, void *stream)
{
    mtp_status st = check_batch(batch);
    if (st != MTP_OK) return st;
    if (batch == 0) return MTP_OK;
    if (!keys || !out_tokens) return MTP_ERR_NULL;
    return cuda_status(launch_decode_keys(keys, batch, out_tokens, out_max, (cudaStream_t)stream));
}

int32_t mtp_gather_plan(const mtp_head_desc *desc, int32_t batch)
{
    mtp_status st = check_desc(desc, true, true, true);
    if (st != MTP_OK) return st;
    st = check_batch(batch);
    if (st != MTP_OK) return st;
    if (batch == 0) return 0;
    int chunk = 0;
    const GatherKind k = gather_kind(desc, batch, false, &chunk);
    return k == kGatherNone ? (int32_t)MTP_ERR_UNSUPPORTED : (int32_t)k;
}

mtp_status mtp_force_gather(int32_t kind)
{
    if (kind < -1 || kind > kGatherFused) return MTP_ERR_SHAPE;
    g_force_kind.store(kind);
    return MTP_OK;
}

mtp_status mtp_wait_test(int64_t limit_ns, int32_t stall)
{
    if (limit_ns < 0) return MTP_ERR_SHAPE;
    g_wait_ns.store(limit_ns == 0 ? kDefaultWaitNs : (unsigned long long)limit_ns);
    g_stall_test.store(stall != 0 ? 1 : 0);
    return MTP_OK;
}

mtp_status mtp_read_device_error(const void *workspace, uint32_t *host_word, void *stream)
{
    if (!workspace || !host_word) return MTP_ERR_NULL;
    return cuda_status(cudaMemcpyAsync(host_word, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                       (cudaStream_t)stream));
}

const char *mtp_status_string(mtp_status status)
{
    switch (status) {
    case MTP_OK: return "ok";
    case MTP_ERR_NULL: return "a required pointer is NULL";
    case MTP_ERR_SHAPE: return "a size is out of range or inconsistent";
    case MTP_ERR_ALIGN: return "a pointer or row stride is not 16-byte aligned";
    case MTP_ERR_WORKSPACE: return "workspace missing or smaller than mtp_workspace_bytes";
    case MTP_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case MTP_ERR_UNSUPPORTED: return "sizes outside the library's limits";
    }
    return "unknown status";
}

int32_t mtp_version(void) { return 100; }

mtp_status mtp_profile_events(int32_t kernel, void *start_event, void *stop_event)
{
    if (kernel < 0 || kernel > MTP_KERNEL_DENSE) return MTP_ERR_SHAPE;
    g_prof[kernel][0] = start_event;
    g_prof[kernel][1] = stop_event;
    return MTP_OK;
}

}  // extern "C"
