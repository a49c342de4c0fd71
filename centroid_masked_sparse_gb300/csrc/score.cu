// Gather + sparse dot products + argmax / scatter.
//
// Steps 3-4 and the two finishes of Gemma4MTPMaskedEmbedder ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py):
// _select_and_score maps each selected centroid to its token ids through
// token_ordering.view(C, V/C), gathers those lm_head rows and dots them with
// the hidden state; get_top_tokens keeps the token id of the largest logit;
// forward scatters the logits into a full-vocabulary row that is -inf
// elsewhere (the -inf fill is a separate kernel that runs first).
//
// Work is cluster-major and deduplicated: a work item is a chunk of one
// selected cluster's ordered positions, together with every batch row that
// selected the cluster (the bucket built by the top-K kernel), so each
// candidate embedding row is read from HBM once per call however many rows
// chose its cluster.
//
// The kernel is a producer/consumer pipeline, one CTA per SM:
//   - one producer warp walks this CTA's share of the work items (records and
//     metadata prefetched two and one items ahead), bulk-copies
//     (cp.async.bulk, the TMA engine) the item's hidden rows into one of four
//     h buffers and every candidate's embedding row (3 KB at H=1536) into a
//     ring of ~50 shared-memory slots, one lane per slot, each completing on
//     its own mbarrier, with an evict-first L2 policy (rows are read once);
//   - 24 consumer warps (16 for H up to 3072, else 8) take slots in turn, dot the
//     row against the item's hidden rows out of shared memory (16-byte lanes,
//     f32 FMAs fed with bf16 halves, a butterfly of shuffles per dot), then
//     either store the logit into the full-vocabulary row or keep the best
//     (logit, lower token id) key per row in a register until the item
//     changes, then fold it into a per-CTA 64-bit shared atomicMax.
// So ~140 KB of candidate rows are in flight per SM without holding a single
// register, which is what the HBM latency-bandwidth product needs.
//
// Barrier phases: a parity wait on an mbarrier is only meaningful while the
// waiter is at most one phase ahead of the barrier.  Slot s carries sequence
// numbers s, s+R, s+2R, ... and consumer warp w takes sequence numbers
// w, w+NW, ...; with R a multiple of NW every phase of a slot goes to the same
// warp, which waits for them in order, so no warp can wait on phase j of a slot
// while phase j-1 is still in flight (and mistake the completed phase j-2 for
// it).  The producer publishes at most min(32, R) consecutive sequence numbers
// at once, so it never holds two phases of one slot either.  The last
// CTA to finish (a ticket, never a wait) turns the per-row keys into token
// ids.  Every mbarrier wait gives up after a wall-clock limit and records
// MTP_DEVERR_TIMEOUT rather than hanging.
#include <algorithm>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace mtp {

using namespace sm100;

namespace {

constexpr int kHBuffers = 4;
constexpr int kMaxRowGroup = 8;
constexpr int kTokDone = -2;

// Sites of a wait that gave up, recorded once per call for diagnosis.
enum WaitSite : uint32_t {
    kSiteConsumerFull = 1,
    kSiteConsumerHFull = 2,
    kSiteConsumerLastHFull = 3,
    kSiteProducerHEmpty = 4,
    kSiteProducerEmpty = 5,
    kSiteProducerDone = 6
};

__device__ __forceinline__ void record_timeout(const GatherParams &p, uint32_t site, uint32_t seq)
{
    atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TIMEOUT);
    if (atomicCAS(p.ctrl + kCtrlWaitSite, 0u, site) == 0u) {
        p.ctrl[kCtrlWaitCta] = blockIdx.x;
        p.ctrl[kCtrlWaitSeq] = seq;
    }
}

struct SlotMeta {
    int tok;      // token id, -1: skipped (invalid id), kTokDone: end of stream
    uint32_t use; // h-buffer use number: buffer use % 4, phase parity (use / 4) & 1
    int pos;      // position of the token inside its cluster (the sparse pair's column)
};

struct HMeta {
    int rows[kMaxRowGroup];
    int ranks[kMaxRowGroup];   // rank of the item's cluster in each row's top-K (sparse pair)
    int gr;       // rows in this group
    int left;     // slots of this item not yet consumed
};

struct Smem {
    uint8_t *ring, *hbuf;
    uint32_t full0, empty0, hfull0, hempty0;
    SlotMeta *meta;
    HMeta *hmeta;
    unsigned long long *best;
    int *prow;   // the producer's row list of the current item [B]
    int *prank;  // rank of the item's cluster in each of those rows' top-K [B] (sparse pair)
};

__device__ __forceinline__ Smem carve(uint8_t *base, const GatherParams &p)
{
    Smem s;
    const size_t rb = (size_t)p.H * 2;
    s.ring = base;
    s.hbuf = base + (size_t)p.ring * rb;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.hbuf + (size_t)kHBuffers * p.row_group * rb);
    s.full0 = smem_u32(bars);
    s.empty0 = s.full0 + 8u * p.ring;
    s.hfull0 = s.empty0 + 8u * p.ring;
    s.hempty0 = s.hfull0 + 8u * kHBuffers;
    s.meta = reinterpret_cast<SlotMeta *>(bars + 2 * p.ring + 2 * kHBuffers);
    s.hmeta = reinterpret_cast<HMeta *>(s.meta + p.ring);
    s.best = reinterpret_cast<unsigned long long *>(s.hmeta + kHBuffers);
    s.prow = reinterpret_cast<int *>(s.best + p.B);
    s.prank = s.prow + p.B;
    return s;
}

// The producer warp's view of one work item; tok0/tok1 and mask are per lane.
struct ItemMeta {
    int valid;      // a real item (index below the item count)
    int c, p0, nvalid;
    int off;        // p0 minus the cluster's first position
    int tok0, tok1; // token ids at positions p0 + lane and p0 + 32 + lane (-1 beyond nvalid)
    uint32_t mask;  // row-mask word `lane` of the cluster (lane < W)
};

// Metadata of an item whose record (cluster, first position) is already in
// registers: the loads issued here are first used one item later, so their
// latency overlaps the current item's copies.
__device__ __forceinline__ void load_item(const GatherParams &p, int2 item, bool valid, int lane,
                                          ItemMeta &m)
{
    m.valid = valid;
    m.c = -1;
    m.p0 = 0;
    m.off = 0;
    m.nvalid = 0;
    m.tok0 = -1;
    m.tok1 = -1;
    m.mask = 0u;
    if (!valid) return;
    int lo = 0, hi = 0;
    if ((unsigned)item.x < (unsigned)p.C && item.y >= 0)
        cluster_range(p.offsets, p.V, p.S, item.x, &lo, &hi, nullptr);
    const int p0 = item.y > hi - lo ? hi : lo + item.y;
    const int nvalid = max(0, min(p.chunk, hi - p0));
    m.c = item.x;
    m.p0 = p0;
    m.off = p0 - lo;
    m.nvalid = nvalid;
    if (nvalid == 0) return;
    if (lane < nvalid) m.tok0 = __ldg(p.ordering + p0 + lane);
    if (lane + kWarp < nvalid) m.tok1 = __ldg(p.ordering + p0 + kWarp + lane);
    if (lane < p.W) m.mask = __ldcg(p.rowmask + (size_t)item.x * p.W + lane);
}

// The next item of a CTA after item it.  Uniform clusters make equal items, so CTA j
// takes j, j + G, j + 2G, ... (an even split without atomics; a hand-out by atomics
// measured slower there).  Ragged clusters make items of unequal cost: after its
// first item a CTA takes a ticket on the call's item counter (cleared with the other
// control words by the projection), so CTAs that finish early take more.
__device__ __forceinline__ int next_item(const GatherParams &p, int it, int lane)
{
    if (p.offsets == nullptr) return it + (int)gridDim.x;
    int nx = 0;
    if (lane == 0) nx = (int)gridDim.x + (int)atomicAdd(p.ctrl + kCtrlNext, 1u);
    return __shfl_sync(0xffffffffu, nx, 0);
}

// Producer warp: walks the items of this CTA (item blockIdx.x, then next_item's) and
// publishes, per
// row group, the hidden rows into an h buffer and one ring slot per candidate
// position (each lane issues its own slot's bulk copy).  The item records and
// their metadata are loaded two and one items ahead.  False after a timed-out wait.
__device__ bool produce(const GatherParams &p, const Smem &sm, int lane, int consumers)
{
    const uint32_t rb = (uint32_t)p.H * 2;
    int it1 = (int)blockIdx.x;
    const int2 invalid_item = make_int2(-1, 0);
    // the first two item records are loaded together with the item count, not after it
    // (both slots lie inside the list; a record past the count is dropped)
    const int2 rec0 = it1 < p.items_cap ? p.items[it1] : invalid_item;
    const int n_items = (int)min(p.ctrl[kCtrlItems], (uint32_t)p.items_cap);
    int it2 = next_item(p, it1, lane);
    const int2 rec1 = it2 < p.items_cap ? p.items[it2] : invalid_item;
    const uint64_t pol = l2_policy_evict_first();
    const int step = p.step;
    const uint32_t ring = (uint32_t)p.ring;
    uint32_t seq = 0, huse = 0;
    uint32_t seq_slot = 0, seq_par = 0;   // slot and phase parity of sequence number `seq`
    ItemMeta nxt;
    load_item(p, it1 < n_items ? rec0 : invalid_item, it1 < n_items, lane, nxt);
    int2 rec2 = it2 < n_items ? rec1 : invalid_item;   // record of the item after next
    for (;;) {
        const ItemMeta cur = nxt;
        if (!cur.valid) break;
        load_item(p, rec2, it2 < n_items, lane, nxt);
        if (it2 < n_items) it2 = next_item(p, it2, lane);
        rec2 = it2 < n_items ? p.items[it2] : invalid_item;
        if (cur.nvalid == 0) continue;
        // the bucket's batch rows, in row order
        const int cnt = __popc(cur.mask);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = incl - cnt;
        for (uint32_t mm = cur.mask; mm; mm &= mm - 1u) sm.prow[pos++] = lane * kWarp + __ffs(mm) - 1;
        const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
        __syncwarp();
        if (p.sparse_width) {
            // the sparse pair's column block of each row: the cluster's rank in its top-K
            for (int r = 0; r < total; ++r) {
                const int32_t *sel = p.topk + (size_t)sm.prow[r] * p.K;
                int rank = -1;
                for (int k0 = 0; k0 < p.K && rank < 0; k0 += kWarp) {
                    const bool hit = k0 + lane < p.K && __ldcg(sel + k0 + lane) == cur.c;
                    const unsigned bal = __ballot_sync(0xffffffffu, hit);
                    if (bal) rank = k0 + __ffs(bal) - 1;
                }
                if (lane == 0) sm.prank[r] = rank;
            }
            __syncwarp();
        }
        for (int g0 = 0; g0 < total; g0 += p.row_group) {
            const int gr = min(p.row_group, total - g0);
            const int hb = (int)(huse % kHBuffers);
            const uint32_t hpar = (huse / kHBuffers) & 1u;
            int ok = 1;
            if (lane == 0) {
                // (the wait test makes the first use wait for the phase that nothing
                // completes: no copy has been issued yet, so the CTA leaves clean)
                const uint32_t stall = (p.stall_test && huse == 0u) ? 1u : 0u;
                ok = mbar_wait(sm.hempty0 + 8u * hb, hpar ^ 1u ^ stall, p.wait_ns);
                if (!ok) record_timeout(p, kSiteProducerHEmpty, huse);
                if (ok) {
                    HMeta &hm = sm.hmeta[hb];
                    for (int r = 0; r < gr; ++r) {
                        hm.rows[r] = sm.prow[g0 + r];
                        if (p.sparse_width) hm.ranks[r] = sm.prank[g0 + r];
                    }
                    hm.gr = gr;
                    hm.left = cur.nvalid;
                    __threadfence_block();
                    mbar_arrive_expect_tx(sm.hfull0 + 8u * hb, (uint32_t)gr * rb);
                }
            }
            // The slots of this use are published by every lane, and consumers read the
            // metadata above once they see a slot: __syncwarp orders lane 0's stores before
            // the other lanes' releases (a shuffle alone would not order memory).
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
            if (lane < gr)
                bulk_copy_g2s(smem_u32(sm.hbuf + ((size_t)hb * p.row_group + lane) * rb),
                              p.hidden + (size_t)sm.prow[g0 + lane] * p.H, rb, sm.hfull0 + 8u * hb);
            ++huse;
            for (int l0 = 0; l0 < cur.nvalid; l0 += step) {
                const int q = l0 + lane;
                const int a = __shfl_sync(0xffffffffu, cur.tok0, q & (kWarp - 1));
                const int b = __shfl_sync(0xffffffffu, cur.tok1, q & (kWarp - 1));
                bool lok = true;
                if (lane < step && q < cur.nvalid) {
                    int tok = q < kWarp ? a : b;
                    if ((unsigned)tok >= (unsigned)p.V) {
                        atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
                        tok = -1;
                    }
                    const uint32_t sq = seq + (uint32_t)q;
                    uint32_t slot = seq_slot + (uint32_t)q, par = seq_par;
                    while (slot >= ring) {   // q < 64: at most a couple of wraps
                        slot -= ring;
                        par ^= 1u;
                    }
                    lok = mbar_wait(sm.empty0 + 8u * slot, par ^ 1u, p.wait_ns);
                    if (!lok) record_timeout(p, kSiteProducerEmpty, sq);
                    if (lok) {
                        sm.meta[slot].tok = tok;
                        sm.meta[slot].use = huse - 1u;
                        sm.meta[slot].pos = cur.off + q;
                        if (tok >= 0) {
                            mbar_arrive_expect_tx(sm.full0 + 8u * slot, rb);
                            bulk_copy_g2s_hint(smem_u32(sm.ring + (size_t)slot * rb),
                                               p.embed + (long long)tok * p.ld, rb, sm.full0 + 8u * slot,
                                               pol);
                        } else {
                            mbar_arrive(sm.full0 + 8u * slot);
                        }
                    }
                }
                if (__any_sync(0xffffffffu, !lok)) return false;
            }
            seq += (uint32_t)cur.nvalid;
            seq_slot += (uint32_t)cur.nvalid;
            while (seq_slot >= ring) {
                seq_slot -= ring;
                seq_par ^= 1u;
            }
        }
    }
    // one end-of-stream marker per consumer warp
    bool ok = true;
    if (lane < consumers) {
        const uint32_t sq = seq + (uint32_t)lane;
        uint32_t slot = seq_slot + (uint32_t)lane, par = seq_par;
        while (slot >= ring) {
            slot -= ring;
            par ^= 1u;
        }
        ok = mbar_wait(sm.empty0 + 8u * slot, par ^ 1u, p.wait_ns);
        if (!ok) record_timeout(p, kSiteProducerDone, sq);
        if (ok) {
            sm.meta[slot].tok = kTokDone;
            sm.meta[slot].use = 0u;
            mbar_arrive(sm.full0 + 8u * slot);
        }
    }
    return !__any_sync(0xffffffffu, !ok);
}

template <int NCH, bool SCATTER, int NW, bool FULL>
__device__ bool consume(const GatherParams &p, const Smem &sm, int warp, int lane)
{
    const uint32_t rb = (uint32_t)p.H * 2;
    const int hv = p.H >> 3;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint32_t ready_use = 0xffffffffu;   // h-buffer use whose rows are known to have landed
    uint32_t best_use = 0xffffffffu;    // use whose argmax this warp holds in registers
    unsigned long long best = 0ull;     // lane r: best key of row best_row of that use
    int best_row = 0;
    bool ok = true;
    // this warp's sequence numbers are warp, warp + NW, ...; with the ring a multiple of
    // NW its slots are warp, warp + NW, ... < ring, then the same slots one phase later
    uint32_t slot = (uint32_t)warp, par = 0u;
    for (uint32_t k = 0;; ++k, slot += NW) {
        if (slot >= (uint32_t)p.ring) {
            slot -= (uint32_t)p.ring;
            par ^= 1u;
        }
        const uint32_t seq = (uint32_t)warp + k * NW;
        if (!mbar_wait(sm.full0 + 8u * slot, par, p.wait_ns)) {
            if (lane == 0) record_timeout(p, kSiteConsumerFull, seq);
            ok = false;
            break;
        }
        const SlotMeta m = sm.meta[slot];
        if (m.tok == kTokDone) break;
        const int hb = (int)(m.use % kHBuffers);
        const uint32_t hpar = (m.use / kHBuffers) & 1u;
        if (!SCATTER && m.use != best_use) {
            // a new item: fold the previous item's per-row bests into the CTA's keys
            if (best) atomicMax(sm.best + best_row, best);
            best = 0ull;
            best_use = m.use;
        }
        // Take the candidate row into registers and hand the slot straight back to the
        // producer: the ring then holds copies in flight, not rows waiting for arithmetic.
        uint4 e[NCH];
        if (m.tok >= 0) {
            const uint4 *erow = reinterpret_cast<const uint4 *>(sm.ring + (size_t)slot * rb);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int idx = c * kWarp + lane;
                e[c] = (FULL || idx < hv) ? erow[idx] : zero;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty0 + 8u * slot);
        if (m.tok >= 0) {
            if (m.use != ready_use) {
                if (!mbar_wait(sm.hfull0 + 8u * hb, hpar, p.wait_ns)) {
                    if (lane == 0) record_timeout(p, kSiteConsumerHFull, m.use);
                    ok = false;
                    break;
                }
                ready_use = m.use;
            }
            const HMeta &hm = sm.hmeta[hb];
            const int gr = hm.gr;
            for (int r = 0; r < gr; ++r) {
                const uint4 *hrow =
                    reinterpret_cast<const uint4 *>(sm.hbuf + ((size_t)hb * p.row_group + r) * rb);
                // four independent chains (one per 32-bit word of a 16-byte group)
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const int idx = c * kWarp + lane;
                    if (FULL || idx < hv) {
                        const uint4 x = hrow[idx];
                        a0 = fma2_bf16(e[c].x, x.x, a0);
                        a1 = fma2_bf16(e[c].y, x.y, a1);
                        a2 = fma2_bf16(e[c].z, x.z, a2);
                        a3 = fma2_bf16(e[c].w, x.w, a3);
                    }
                }
                float acc = warp_sum((a0 + a1) + (a2 + a3));
                if (p.bf16_logits) acc = round_bf16(acc);
                if (lane == r) {
                    const int row = hm.rows[r];
                    if (SCATTER) {
                        if (p.sparse_width) {
                            const int rank = hm.ranks[r];
                            if (rank >= 0) {
                                const size_t o = (size_t)row * p.sparse_width + (size_t)rank * p.S + m.pos;
                                p.out_logits[o] = acc;
                                if (p.out_ids) p.out_ids[o] = m.tok;
                            }
                        } else {
                            p.out_logits[(size_t)row * p.V + m.tok] = acc;
                        }
                    } else {
                        const unsigned long long key = argmax_key(acc, m.tok);
                        best = key > best ? key : best;
                        best_row = row;
                    }
                }
            }
        }
        // for the item's last slot, release its h buffer once its hidden rows have landed
        // (a skipped slot never waited for them)
        __syncwarp();
        if (lane == 0 && atomicSub(&sm.hmeta[hb].left, 1) == 1) {
            if (!mbar_wait(sm.hfull0 + 8u * hb, hpar, p.wait_ns)) {
                record_timeout(p, kSiteConsumerLastHFull, m.use);
                ok = false;
            }
            mbar_arrive(sm.hempty0 + 8u * hb);
        }
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
    }
    if (!SCATTER && best) atomicMax(sm.best + best_row, best);
    return ok;
}

template <int NCH, bool SCATTER, int NW, bool FULL>
__global__ void __launch_bounds__((NW + 1) * kWarp, NW >= 16 ? 1 : 2) k_gather_score(const GatherParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_last;
    constexpr int kThreads = (NW + 1) * kWarp;
    const Smem sm = carve(smem, p);
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x & (kWarp - 1);

    if (p.ring % NW != 0 || p.consumer_warps != NW || p.step > p.ring || p.step > kWarp) {
        // a slot shared by two consumer warps could be waited one phase early: refuse
        if (threadIdx.x == 0) atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TIMEOUT);
        return;
    }
    if (threadIdx.x == 0) {
        for (int r = 0; r < p.ring; ++r) {
            mbar_init(sm.full0 + 8u * r, 1);
            mbar_init(sm.empty0 + 8u * r, 1);
        }
        for (int b = 0; b < kHBuffers; ++b) {
            mbar_init(sm.hfull0 + 8u * b, 1);
            mbar_init(sm.hempty0 + 8u * b, 1);
        }
        fence_barrier_init();
    }
    if (!SCATTER)
        for (int b = threadIdx.x; b < p.B; b += kThreads) sm.best[b] = 0ull;
    __syncthreads();
    prefetch_l2_table(p.ordering, (size_t)p.V * sizeof(int32_t));
    prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    // the work items, row masks and counters come from the top-K kernel before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");

    bool ok = true;
    if (warp == NW) {
        ok = produce(p, sm, lane, NW);
    } else {
        ok = consume<NCH, SCATTER, NW, FULL>(p, sm, warp, lane);
    }
    if (!ok && lane == 0) atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TIMEOUT);
    __syncthreads();

    if (SCATTER) return;
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
        const unsigned long long k = sm.best[b];
        if (k) atomicMax(p.keys + b, k);
    }
    // the last CTA to finish turns the keys into token ids
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

template <int NCH, bool SCATTER, int NW, bool FULL>
cudaError_t run_gather_nw(const GatherParams &p, cudaStream_t s)
{
    const void *fn = (const void *)k_gather_score<NCH, SCATTER, NW, FULL>;
    const size_t smem = gather_smem_bytes(p);
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(k_gather_score<NCH, SCATTER, NW, FULL>, dim3(sm_count() * p.ctas_per_sm),
                            dim3((NW + 1) * kWarp), smem, s, p);
}

// Consumer warps: 24 while the row registers allow it (H <= 2048), 16 up to H = 3072,
// else 8; FULL when H is a whole number of 256-element chunks (no tail lanes).
template <int NCH, bool SCATTER>
cudaError_t run_gather(const GatherParams &p, cudaStream_t s)
{
    const bool full = p.H == NCH * 256;
    constexpr int NW = NCH <= 8 ? 24 : (NCH <= 12 ? 16 : 8);
    if (p.consumer_warps == NW)
        return full ? run_gather_nw<NCH, SCATTER, NW, true>(p, s) : run_gather_nw<NCH, SCATTER, NW, false>(p, s);
    return cudaErrorInvalidValue;
}

template <bool SCATTER>
cudaError_t dispatch_gather(const GatherParams &p, cudaStream_t s)
{
    switch (chunks_for_hidden(p.H)) {
    case 1: return run_gather<1, SCATTER>(p, s);
    case 2: return run_gather<2, SCATTER>(p, s);
    case 3: return run_gather<3, SCATTER>(p, s);
    case 4: return run_gather<4, SCATTER>(p, s);
    case 5: return run_gather<5, SCATTER>(p, s);
    case 6: return run_gather<6, SCATTER>(p, s);
    case 8: return run_gather<8, SCATTER>(p, s);
    case 10: return run_gather<10, SCATTER>(p, s);
    case 12: return run_gather<12, SCATTER>(p, s);
    case 16: return run_gather<16, SCATTER>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t gather_smem_bytes(const GatherParams &p)
{
    const size_t rb = (size_t)p.H * 2;
    return (size_t)p.ring * rb + (size_t)kHBuffers * p.row_group * rb +
           (size_t)(2 * p.ring + 2 * kHBuffers) * 8 + (size_t)p.ring * sizeof(SlotMeta) +
           kHBuffers * sizeof(HMeta) + (size_t)p.B * 16;
}

// Geometry of the gather kernel for p.H and p.B: consumer warps, CTAs per SM,
// ring slots, hidden rows per h buffer and the producer's batch width.  The ring
// is a multiple of the consumer warp count, so each slot always belongs to the
// same warp (see the kernel's comment on barrier phases).
void gather_geometry(GatherParams &p)
{
    const size_t rb = (size_t)p.H * 2;
    const int nch = chunks_for_hidden(p.H);
    p.consumer_warps = nch <= 8 ? 24 : (nch <= 12 ? 16 : 8);
    p.ctas_per_sm = 1;
    int rg = (int)(16384 / rb);
    rg = rg < 1 ? 1 : (rg > kMaxRowGroup ? kMaxRowGroup : rg);
    if (rg > p.B) rg = p.B;
    p.row_group = rg;
    const size_t budget = (size_t)(212 * 1024) / (size_t)p.ctas_per_sm;
    const size_t fixed = (size_t)kHBuffers * rg * rb + kHBuffers * (sizeof(HMeta) + 16) + (size_t)p.B * 16 + 64;
    long long r = fixed < budget ? (long long)((budget - fixed) / (rb + 16 + sizeof(SlotMeta))) : 0;
    const int nw = p.consumer_warps;
    if (r > 256) r = 256;
    r = r / nw * nw;
    if (r < nw) r = nw;
    p.ring = (int)r;
    p.step = p.ring < kWarp ? p.ring : kWarp;
}

cudaError_t launch_gather(const GatherParams &p, bool scatter, cudaStream_t s)
{
    return scatter ? dispatch_gather<true>(p, s) : dispatch_gather<false>(p, s);
}

// forward's fill: every entry of the [B, V] row block is -inf before the
// scatter writes the candidates' logits.
// The scatter's background: -inf, or bf16's finite minimum under the fidelity option.
__global__ void __launch_bounds__(256) k_fill(float *out, size_t n, float value)
{
    // the projection and top-K that follow never read this buffer: let them start now
    // (the projection waits for this kernel before it exits, so the gather, which runs
    // after the top-K, writes into a finished fill)
    asm volatile("griddepcontrol.launch_dependents;");
    const float ninf = value;
    const float4 v = make_float4(ninf, ninf, ninf, ninf);
    float4 *o4 = reinterpret_cast<float4 *>(out);
    const size_t n4 = n / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x)
        o4[i] = v;
    if (blockIdx.x == 0 && threadIdx.x < (n & 3))
        out[n4 * 4 + threadIdx.x] = ninf;
}

// Argmax keys as signed-comparable int64 (the sign bit flipped: unsigned order
// becomes signed order, and the empty key 0 becomes INT64_MIN), and back.
__global__ void k_export_keys(const unsigned long long *keys, int B, int64_t *out)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) out[b] = (int64_t)(__ldcg(keys + b) ^ 0x8000000000000000ull);
}

__global__ void k_decode_keys(const int64_t *keys, int B, int32_t *tokens, float *maxv)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int32_t tok;
    float v;
    decode_argmax_key((unsigned long long)keys[b] ^ 0x8000000000000000ull, &tok, &v);
    tokens[b] = tok;
    if (maxv) maxv[b] = v;
}

cudaError_t launch_export_keys(const unsigned long long *keys, int B, int64_t *out, cudaStream_t s)
{
    k_export_keys<<<(B + 255) / 256, 256, 0, s>>>(keys, B, out);
    return cudaGetLastError();
}

cudaError_t launch_decode_keys(const int64_t *keys, int B, int32_t *tokens, float *maxv, cudaStream_t s)
{
    k_decode_keys<<<(B + 255) / 256, 256, 0, s>>>(keys, B, tokens, maxv);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Direct variant for small batches (at most kDirectMaxB rows): every warp takes one
// candidate at a time, as (work item, position) pairs dealt round-robin over all
// warps of the grid, loads its embedding row straight into registers (16 bytes per
// lane per 256 elements, all in flight at once) and dots it with the bucket's hidden
// rows, which each CTA keeps in shared memory.  No producer and no ring: with few
// candidate rows per SM the pipelined gather's time is its chain of latencies (item
// record, metadata, copy, hand-off), and here a row costs one load round trip, with
// tens of rows in flight per SM.  Same results as the pipelined kernel up to the
// summation order of each dot product; the sparse pair is not done here.
// ---------------------------------------------------------------------------
constexpr int kDirectThreads = 256;
constexpr int kDirectMaxB = 32;   // one row-mask word

template <int NCH, bool SCATTER>
__global__ void __launch_bounds__(kDirectThreads) k_gather_direct(const GatherParams p)
{
    extern __shared__ uint4 hsm[];   // [B][H / 8] hidden rows
    __shared__ unsigned long long s_best[kDirectMaxB];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & (kWarp - 1), warp = tid / kWarp;
    const int hv = p.H >> 3;
    if (!SCATTER && tid < kDirectMaxB) s_best[tid] = 0ull;
    prefetch_l2_table(p.ordering, (size_t)p.V * sizeof(int32_t));
    prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    // the items and buckets come from the top-K kernel before this one (and the hidden
    // rows, with host-resident input, from the staging kernel before that)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < p.B * hv; i += kDirectThreads) hsm[i] = ld_ro16(p.hidden + (size_t)i * 8);
    __syncthreads();

    const int n_items = (int)min(p.ctrl[kCtrlItems], (uint32_t)p.items_cap);
    const int n_cand = n_items * p.chunk;
    const int nwarps = (int)gridDim.x * (kDirectThreads / kWarp);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

    for (int cand = (int)blockIdx.x * (kDirectThreads / kWarp) + warp; cand < n_cand; cand += nwarps) {
        const int it = cand / p.chunk, pos = cand - it * p.chunk;
        const int2 rec = p.items[it];
        // a slot the top-K left unwritten (an append it dropped with overlapping offsets)
        // holds stale data: such records are skipped, never followed
        if ((unsigned)rec.x >= (unsigned)p.C || rec.y < 0) continue;
        int lo, hi;
        if (!cluster_range(p.offsets, p.V, p.S, rec.x, &lo, &hi, p.ctrl + kCtrlError)) continue;
        const int at = (rec.y > hi - lo ? hi : lo + rec.y) + pos;
        if (at >= hi) continue;   // past the end of a tail chunk
        const int tok = __ldg(p.ordering + at);
        if ((unsigned)tok >= (unsigned)p.V) {
            if (lane == 0) atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
            continue;
        }
        uint32_t mask = __ldcg(p.rowmask + (size_t)rec.x * p.W);   // B <= 32: one word
        const uint16_t *row = p.embed + (size_t)tok * p.ld;
        uint4 e[NCH];
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int idx = k * kWarp + lane;
            e[k] = idx < hv ? ld_stream16(row + (size_t)idx * 8) : zero;
        }
        while (mask) {
            const int b = __ffs(mask) - 1;
            mask &= mask - 1u;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
                const int idx = k * kWarp + lane;
                if (idx < hv) acc = dot8_bf16_mixed(e[k], hsm[b * hv + idx], acc);
            }
            acc = warp_sum(acc);
            if (p.bf16_logits) acc = round_bf16(acc);
            if (SCATTER) {
                if (lane == 0) p.out_logits[(size_t)b * p.V + tok] = acc;
            } else if (lane == 0) {
                atomicMax(&s_best[b], argmax_key(acc, tok));   // the CTA's best per row
            }
        }
    }
    if (SCATTER) return;
    __syncthreads();
    if (tid < p.B && s_best[tid]) atomicMax(p.keys + tid, s_best[tid]);
    // the last CTA to finish turns the keys into token ids
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(p.ctrl + kCtrlTicket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < p.B) {
        const unsigned long long k = atomicAdd(p.keys + tid, 0ull);
        int32_t t;
        float v;
        decode_argmax_key(k, &t, &v);
        p.out_tokens[tid] = t;
        if (p.out_max) p.out_max[tid] = v;
    }
}

template <int NCH, bool SCATTER>
cudaError_t run_gather_direct(const GatherParams &p, cudaStream_t s)
{
    const size_t smem = (size_t)p.B * (size_t)(p.H / 8) * sizeof(uint4);
    const void *fn = (const void *)k_gather_direct<NCH, SCATTER>;
    cudaError_t e = allow_smem(fn, smem);
    if (e != cudaSuccess) return e;
    const int per_sm = std::max(1, std::min(8, blocks_per_sm(fn, kDirectThreads, smem)));
    return launch_dependent(k_gather_direct<NCH, SCATTER>, dim3((unsigned)(per_sm * sm_count())),
                            dim3(kDirectThreads), smem, s, p);
}

template <bool SCATTER>
cudaError_t dispatch_gather_direct(const GatherParams &p, cudaStream_t s)
{
    switch (chunks_for_hidden(p.H)) {
    case 1: return run_gather_direct<1, SCATTER>(p, s);
    case 2: return run_gather_direct<2, SCATTER>(p, s);
    case 3: return run_gather_direct<3, SCATTER>(p, s);
    case 4: return run_gather_direct<4, SCATTER>(p, s);
    case 5: return run_gather_direct<5, SCATTER>(p, s);
    case 6: return run_gather_direct<6, SCATTER>(p, s);
    case 8: return run_gather_direct<8, SCATTER>(p, s);
    case 10: return run_gather_direct<10, SCATTER>(p, s);
    case 12: return run_gather_direct<12, SCATTER>(p, s);
    case 16: return run_gather_direct<16, SCATTER>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gather_direct(const GatherParams &p, bool scatter, cudaStream_t s)
{
    if (p.B < 1 || p.B > kDirectMaxB || p.W != 1 || p.chunk < 1 || p.sparse_width) return cudaErrorInvalidValue;
    return scatter ? dispatch_gather_direct<true>(p, s) : dispatch_gather_direct<false>(p, s);
}

// Copy of the batch's hidden rows from memory the device reads over the host link
// (pinned host memory) into the workspace: one 16-byte load per thread and round,
// all of them in flight at once, so the copy costs about one link round trip.
__global__ void __launch_bounds__(256) k_stage_rows(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                                    size_t n16)
{
    // the projection behind it starts now and waits for this kernel before it reads the rows
    asm volatile("griddepcontrol.launch_dependents;");
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_stage_rows(void *dst, const void *src, size_t bytes, cudaStream_t s)
{
    if ((bytes & 15) || ((uintptr_t)dst & 15) || ((uintptr_t)src & 15)) return cudaErrorInvalidValue;
    const size_t n16 = bytes / 16;
    if (n16 == 0) return cudaSuccess;
    const size_t blocks = std::min<size_t>((n16 + 255) / 256, (size_t)sm_count());
    k_stage_rows<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<uint4 *>(dst),
                                                 reinterpret_cast<const uint4 *>(src), n16);
    return cudaGetLastError();
}

cudaError_t launch_fill(float *out, size_t n, float value, cudaStream_t s)
{
    // two CTAs per SM: enough stores in flight for the write stream, and room left on
    // every SM for the projection and top-K that start behind it
    k_fill<<<sm_count() * 2, 256, 0, s>>>(out, n, value);
    return cudaGetLastError();
}

}  // namespace mtp
