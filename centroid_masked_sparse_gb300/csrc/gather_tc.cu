// Gather + sparse dot products on the tensor cores.
//
// Steps 3-4 and both finishes of Gemma4MTPMaskedEmbedder ("Add Gemma4 MTP
// speculative decoding with centroids masking", vLLM gemma4_mtp.py), like
// score.cu, but each work item is treated as the small dense contraction it is:
// logits[t, r] = sum_k E[tok_t, k] * h[row_r, k] for the item's candidate
// positions t (at most 128) and the rows r of the cluster's bucket.
//
// One unit = (work item, block of at most nmax bucket rows).  The candidate
// embedding rows are the MMA's M side (one token per TMEM lane, M = 128 with the
// lanes past the chunk ignored), the bucket's hidden rows its N side (padded to
// a multiple of 16), K = H in 64-element blocks.  With the packed table and
// clusters of at most 64 positions on average, two chunks of at most 64
// candidates whose buckets together fit share a unit (tile rows 0-63 and 64-127,
// the union of the buckets as N; the epilogue keeps a pair only where the row
// selected that candidate's cluster): a separate instantiation (PAIR).  Operands reach shared memory
// by TMA in the 128-byte-swizzled layout the MMA descriptors expect:
//   * with the packed embedding table (below) the chunk's candidate rows are one
//     or two contiguous, pre-swizzled runs of a 16 KB block per k-block, fetched
//     with plain bulk copies that stop at the chunk's last real row (a cluster's
//     padding is never read): few large copies are what streams HBM fastest;
//   * with the token-order table they are gathered four rows per instruction
//     (tile::gather4), skipping groups that are all padding;
//   * a small bucket's hidden rows (at most kGatherRowsMax) come by tile::gather4
//     with the A tile, only the groups of four that hold real rows (a padding row
//     inside such a group uses an out-of-range row, which TMA fills with zeros);
//   * a larger bucket's rows are copied by four B warps from L2 (the whole batch
//     stays there) with 16-byte cp.async into the swizzled tile: a gather4 costs
//     the TMA unit far more time than its 512 bytes suggest, so with many rows
//     per bucket the count of gathers, not bytes, would set the pace.
// Tile rows that no load wrote hold stale data, which only feeds TMEM lanes and
// columns the epilogue ignores.
//
// Warp roles per CTA (352 threads; two or three CTAs per SM where their TMEM and
// shared memory fit, three with units of at most 32 bucket rows, else one):
//   warp 4   metadata: walks this CTA's items (round-robin; with large buckets
//            by ticket, the next item claimed once the previous one's units are
//            consumed) and publishes each unit's token and row lists into a ring
//            of kMeta entries, running ahead of the loads so that its dependent
//            global reads (item record, row mask, token ids) never stall the
//            stream;
//   warp 6   TMA issue: per unit and k-block, one stage of A loads (and B for a
//            small bucket);
//   warps 7-10 B: the hidden rows of larger buckets, by cp.async (see load_b);
//   warp 5   one thread issues tcgen05.mma (kind::f16, fp32 in TMEM, four
//            accumulators so the epilogues of the last units overlap the next);
//   warps 0-3 epilogue: tcgen05.ld of the unit's logits (thread = candidate),
//            then the scatter store or the per-row argmax fold (a reduce-scatter
//            butterfly over the warp's candidates for each group of columns).
// Every mbarrier wait is bounded and records MTP_DEVERR_TIMEOUT if it gives up.
//
// The packed table (its layout is specified with mtp_pack_embeddings in the C
// header) stores each cluster's rows in ordered-position order, padded to 32
// rows, as 16 KB blocks of 128 padded rows x 64 elements in the 128-byte
// swizzle.  A run of rows starting at a multiple of 8 rows, copied to a
// 1024-byte-aligned stage, is already the MMA's K-major operand (the swizzle
// depends on the row modulo 8 only).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <climits>
#include <mutex>
#include <map>
#include <tuple>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace mtp {

using namespace sm100;

namespace {

constexpr int kBWarps = 4;         // warps that copy the buckets' hidden rows (the B operand)
constexpr int kThreads = (7 + kBWarps) * kWarp;
constexpr int kTileM = 128;        // MMA M: candidate positions per unit (at most)
constexpr int kTileK = 64;         // bf16 per k-block (128-byte rows)
constexpr int kMaxN = 64;          // bucket rows per unit (at most): with four accumulators a CTA
                                   // then takes at most half the TMEM, so two CTAs fit on an SM
                                   // (three with the 32-row units of calls with small buckets)
constexpr int kMeta = 8;           // unit-metadata ring
constexpr int kAcc = 4;            // TMEM accumulators (at most): the epilogues of the last units overlap the MMAs
constexpr int kMaxStages = 32;
constexpr uint32_t kSmTmemCols = 512;  // TMEM columns of one SM
constexpr uint32_t kRowBytes = kTileK * 2;
constexpr uint32_t kFullABytes = kTileM * kRowBytes;   // what one M = 128 MMA reads
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kMetaReaders = 6 + kBWarps;   // epilogue warps, MMA thread, TMA warp, B warps
constexpr int kBRowsPerThread = kMaxN / (kBWarps * kWarp / 8);   // 8 threads per 128-byte row slice
constexpr int kBLag = 6;               // B copy groups in flight before a stage is signalled full
constexpr int kGatherRowsMax = 8;      // buckets up to this size: B by TMA gather4 (at most two), not the B warps
constexpr int kNoPos = INT_MIN;        // a candidate slot past the chunk's end
constexpr int kPackRows = 32;          // clusters are padded to multiples of this
constexpr int kPackSuper = 128;        // rows per packed block
constexpr uint32_t kPackBlock = kPackSuper * kRowBytes;  // 16384 bytes

struct UnitMeta {
    int tok[kTileM];    // candidate token ids (-1: padding or invalid id)
    int rows[kMaxN];    // bucket rows of this unit (n of them), then p.B up to npad
    int n;              // rows in this unit; -1: end of stream
    int npad, nvalid;
    int p0;             // token-order table: first ordered position; packed: first group
    int local0;         // position of the chunk's first candidate inside its cluster
    int g1, nvalid1;    // a paired unit's second chunk (packed: first group, candidates)
    int ranks[kMaxN];   // sparse pair: rank of the cluster in each row's top-K
    // per row: bit 0 = a row of the first chunk's bucket, bit 1 = of the second chunk's
    // (the candidates in tile rows 64..127 of a paired unit); 3 for an unpaired unit
    uint8_t half[kMaxN];
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
    int sparse_width;         // sparse pair: row stride K*S of out_logits / out_ids; 0 otherwise
    int bf16_logits;          // logits rounded to bf16 before they are stored or compared
    int32_t *out_ids;
    const int32_t *topk;      // [B, K]
    int K;
    const uint16_t *hidden;   // [B, H]
    int b_lag;                // B copy groups a B thread keeps in flight (<= kBLag, < stages - 1)
    int B, H, V, S, W, C;
    int chunk;      // positions per work item (<= 128; a multiple of 32 when packed)
    const uint8_t *packed;    // packed table blocks, or null (token-order gathers)
    const int32_t *poff;      // its padded cluster offsets [C+1]
    int nmax;       // bucket rows per unit (multiple of 16, <= kMaxN)
    int handout;    // items past the first round by ticket (large buckets), else round-robin
    int num_kb;
    int stages;
    int n_acc;      // TMEM accumulators in use (2 or kAcc)
    uint32_t a_bytes, b_bytes;   // stage sizes
    uint32_t tmem_cols;
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

// Rows of a bucket in row order, block `blk` (nmax rows per block), from the
// bucket's row mask (word `lane` in w): the warp writes them to `rows` and returns
// how many (all lanes).
__device__ int bucket_rows(const Params &p, uint32_t w, int blk, int lane, int *rows)
{
    const int cnt = __popc(w);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int pos = incl - cnt;
    const int lo = blk * p.nmax, hi = lo + p.nmax;
    for (uint32_t m = w; m; m &= m - 1u, ++pos)
        if (pos >= lo && pos < hi) rows[pos - lo] = lane * kWarp + __ffs(m) - 1;
    const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
    return max(0, min(p.nmax, total - lo));
}

// Rows of the union of two buckets (row-mask words wa, wb of this lane) in row order
// (at most nmax), and for each which bucket holds it (bit 0: a, bit 1: b).
__device__ int union_rows(const Params &p, uint32_t wa, uint32_t wb, int lane, int *rows, uint8_t *half)
{
    const uint32_t w = wa | wb;
    const int cnt = __popc(w);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int pos = incl - cnt;
    for (uint32_t m = w; m; m &= m - 1u, ++pos) {
        if (pos >= p.nmax) break;
        const int bit = __ffs(m) - 1;
        rows[pos] = lane * kWarp + bit;
        half[pos] = (uint8_t)(((wa >> bit) & 1u) | (((wb >> bit) & 1u) << 1));
    }
    return min(p.nmax, __shfl_sync(0xffffffffu, incl, kWarp - 1));
}

__device__ __forceinline__ int warp_count(uint32_t w)
{
    int c = __popc(w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
}

// The metadata warp's view of one work item: its range and the loads its units
// need (this lane's row-mask word and token ids, the packed group), issued one
// item before they are used so that their latency overlaps the current item.
struct ItemPre {
    int valid;      // a real item with candidates
    int c, y, lo, p0, nvalid, g0;
    uint32_t w;     // row-mask word `lane` of the cluster
    int tok[kTileM / kWarp];   // token ids at positions p0 + j*32 + lane (kNoPos beyond nvalid)
};

__device__ __forceinline__ void load_item(const Params &p, int2 rec, bool have, int lane, ItemPre &m)
{
    m.valid = 0;
    m.c = rec.x;
    m.y = rec.y;
    m.lo = m.p0 = m.nvalid = m.g0 = 0;
    m.w = 0u;
#pragma unroll
    for (int j = 0; j < kTileM / kWarp; ++j) m.tok[j] = kNoPos;
    if (!have) return;
    int lo = 0, hi = 0;
    if ((unsigned)rec.x < (unsigned)p.C && rec.y >= 0)
        cluster_range(p.offsets, p.V, p.S, rec.x, &lo, &hi, nullptr);
    const int p0 = rec.y > hi - lo ? hi : lo + rec.y;
    const int nvalid = max(0, min(p.chunk, hi - p0));
    m.lo = lo;
    m.p0 = p0;
    m.nvalid = nvalid;
    if (nvalid == 0) return;
    m.valid = 1;
    if (lane < p.W) m.w = __ldcg(p.rowmask + (size_t)rec.x * p.W + lane);
#pragma unroll
    for (int j = 0; j < kTileM / kWarp; ++j) {
        const int t = j * kWarp + lane;
        if (t < nvalid) m.tok[j] = __ldg(p.ordering + p0 + t);
    }
    // packed table: the chunk starts at padded position poff[c] + y, a group boundary
    if (p.packed) m.g0 = (__ldg(p.poff + rec.x) + rec.y) / kPackRows;
}

// Candidate token ids of an item for the unit's tile rows lane, lane+32, ... (the item's
// position j*32+lane), -1 past its chunk or for an id outside [0, V) (reported).
__device__ __forceinline__ int unit_token(const Params &p, int tok)
{
    if (tok == kNoPos) return -1;
    if ((unsigned)tok >= (unsigned)p.V) {
        atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
        return -1;
    }
    return tok;
}

// A chunk of at most 64 candidates as the pairing needs it (per lane: row-mask word
// `lane`, token ids of positions lane and 32 + lane).
struct ShortChunk {
    uint32_t w;
    int tok0, tok1, nvalid, g0;
};

__device__ __forceinline__ ShortChunk short_chunk(const ItemPre &m)
{
    return ShortChunk{m.w, m.tok[0], m.tok[1], m.nvalid, m.g0};
}

// Publishes one unit holding chunk a and its whole bucket (at most nmax rows) or, with
// b, chunks a and b together: a's candidates in tile rows 0..63, b's in 64..127, the
// union of their buckets as the unit's rows.  Both chunks are at most 64 candidates
// and the union at most nmax rows (the caller checks).  Packed table only (no sparse
// pair).  False after a timed-out wait.
__device__ bool publish_joint(const Params &p, UnitMeta *meta, uint32_t mfull0, uint32_t mempty0, int &u,
                              int lane, const ShortChunk &a, const ShortChunk *b)
{
    const int um = u % kMeta;
    if (!mbar_wait(mempty0 + 8u * um, ((uint32_t)(u / kMeta) & 1u) ^ 1u, kWaitNs)) return false;
    UnitMeta &m = meta[um];
    const int n = union_rows(p, a.w, b ? b->w : a.w, lane, m.rows, m.half);
    const int npad = (n + 15) & ~15;
    for (int r = n + lane; r < npad; r += kWarp) {
        m.rows[r] = p.B;   // zero rows
        m.half[r] = 0;
    }
    m.tok[lane] = unit_token(p, a.tok0);
    m.tok[kWarp + lane] = unit_token(p, a.tok1);
    m.tok[2 * kWarp + lane] = unit_token(p, b ? b->tok0 : kNoPos);
    m.tok[3 * kWarp + lane] = unit_token(p, b ? b->tok1 : kNoPos);
    if (lane == 0) {
        m.n = n;
        m.npad = npad;
        m.nvalid = a.nvalid;
        m.local0 = 0;
        m.p0 = a.g0;
        m.g1 = b ? b->g0 : 0;
        m.nvalid1 = b ? b->nvalid : 0;
    }
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();
        mbar_arrive(mfull0 + 8u * um);
    }
    ++u;
    return true;
}

// The item a CTA takes after item `prev`.  With large buckets (p.handout): a ticket on
// the call's item counter (cleared with the other control words by the projection),
// offset by the grid, so every item past the first round goes to whichever CTA asks
// first; such items differ in cost (a large bucket is several units), so CTAs that
// finish early take more.  The ticket is taken when the item is about to be needed
// (taking it earlier, to hide the atomic's round trip, measured worse: it leaves fewer
// items to even out the tail).  Otherwise every item is about one unit and the CTAs
// take items prev + G, prev + 2G, ... with no atomic (with tickets, every CTA asking at
// once, the launch took 88.9 instead of 82.9 us on uniform clusters at B=64).
__device__ __forceinline__ int grab_item(const Params &p, int prev, int lane)
{
    if (!p.handout) return prev + (int)gridDim.x;
    int it = 0;
    if (lane == 0) it = (int)gridDim.x + (int)atomicAdd(p.ctrl + kCtrlNext, 1u);
    return __shfl_sync(0xffffffffu, it, 0);
}

// Metadata warp: publishes the units of this CTA's items, pairing short chunks where the
// call allows it, then an end-of-stream entry.  Round-robin (item blockIdx.x, then + G,
// + 2G, ...): item records two items ahead, their loads one item ahead.  Ticketed
// (p.handout): the CTA claims its next item only once the units before the current
// item's are consumed, so it holds at most one item beyond the one in flight; the
// claim, its record and its loads (~2 us) overlap the current item's units.  (Claiming
// as far ahead as the 8-entry metadata ring allowed left CTAs with 2 to 5 units of the
// shared-centroid workload, the slowest ~30 us behind the fastest.)  False after a
// timed-out wait.
template <bool PAIR>
__device__ bool publish_units(const Params &p, UnitMeta *meta, uint32_t mfull0, uint32_t mempty0, int lane)
{
    const int2 none = make_int2(-1, 0);
    int it = blockIdx.x;
    // this CTA's first item record is loaded together with the item count, not after it
    // (the slot lies inside the list; a record past the count is dropped)
    const int2 rec0 = it < p.items_cap ? p.items[it] : none;
    const int n_items = (int)min(p.ctrl[kCtrlItems], (uint32_t)p.items_cap);
    const long long packed_groups = p.packed ? __ldg(p.poff + p.C) / kPackRows : 0;
    int u = 0;
    ShortChunk pend{};         // a chunk of at most 64 candidates waiting for a partner
    bool have_pend = false;
    // publishes the units of one item (or holds a short chunk for a partner)
    auto publish_item = [&](const ItemPre &cur) -> bool {
        if (!cur.valid) return true;
        const int nvalid = cur.nvalid, p0 = cur.p0, g0 = cur.g0;
        // a chunk reaching past the packed table's last group (a table packed from other
        // offsets) is skipped and flagged instead of read
        if (p.packed && (long long)g0 + (nvalid + kPackRows - 1) / kPackRows > packed_groups) {
            if (lane == 0) atomicOr(p.ctrl + kCtrlError, MTP_DEVERR_OFFSETS);
            return true;
        }
        if (PAIR) {
            // two chunks of at most 64 candidates whose buckets together fit a unit share
            // it: the next such item waits here for a partner
            if (nvalid <= kTileM / 2 && warp_count(cur.w) <= p.nmax) {
                const ShortChunk sc = short_chunk(cur);
                if (!have_pend) {
                    pend = sc;
                    have_pend = true;
                    return true;
                }
                const bool fits = warp_count(pend.w | sc.w) <= p.nmax;
                if (!publish_joint(p, meta, mfull0, mempty0, u, lane, pend, fits ? &sc : nullptr)) return false;
                if (fits) {
                    have_pend = false;
                } else {
                    pend = sc;
                }
                return true;
            }
            if (have_pend) {
                if (!publish_joint(p, meta, mfull0, mempty0, u, lane, pend, nullptr)) return false;
                have_pend = false;
            }
        }
        for (int blk = 0;; ++blk) {
            const int um = u % kMeta;
            // a slot acquired for a block that turns out empty is reused by the next
            // unit: its phase is unchanged until a unit is published in it
            if (!mbar_wait(mempty0 + 8u * um, ((uint32_t)(u / kMeta) & 1u) ^ 1u, kWaitNs)) return false;
            UnitMeta &m = meta[um];
            const int n = bucket_rows(p, cur.w, blk, lane, m.rows);
            if (n == 0) break;
            const int npad = (n + 15) & ~15;
            for (int r = n + lane; r < npad; r += kWarp) m.rows[r] = p.B;   // zero rows
            if (PAIR)
                for (int r = lane; r < npad; r += kWarp) m.half[r] = r < n ? 3 : 0;
#pragma unroll
            for (int j = 0; j < kTileM / kWarp; ++j) m.tok[j * kWarp + lane] = unit_token(p, cur.tok[j]);
            if (p.sparse_width) {
                // the sparse pair's column block of each row: the cluster's rank in its top-K
                __syncwarp();   // every lane's row entries are written
                for (int r = 0; r < n; ++r) {
                    const int32_t *sel = p.topk + (size_t)m.rows[r] * p.K;
                    int rank = -1;
                    for (int k0 = 0; k0 < p.K && rank < 0; k0 += kWarp) {
                        const bool hit = k0 + lane < p.K && __ldcg(sel + k0 + lane) == cur.c;
                        const unsigned bal = __ballot_sync(0xffffffffu, hit);
                        if (bal) rank = k0 + __ffs(bal) - 1;
                    }
                    if (lane == 0) m.ranks[r] = rank;
                }
            }
            if (lane == 0) {
                m.n = n;
                m.npad = npad;
                m.nvalid = nvalid;
                m.local0 = p0 - cur.lo;
                m.p0 = p.packed ? g0 : p0;
                if (PAIR) {
                    m.g1 = 0;
                    m.nvalid1 = 0;
                }
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                mbar_arrive(mfull0 + 8u * um);
            }
            ++u;
            if (n < p.nmax) break;   // the bucket ended in this block
        }
        return true;
    };
    if (p.handout) {
        ItemPre cur;
        load_item(p, it < n_items ? rec0 : none, it < n_items, lane, cur);
        while (it < n_items) {
            const int u0 = u;
            if (!publish_item(cur)) return false;
            // the units before this item's are consumed (unit u0 - 1's slot is not reused
            // before unit u0 - 1 + kMeta, so its phase is unambiguous)
            if (u0 > 0 && u > u0 && u - u0 < kMeta &&
                !mbar_wait(mempty0 + 8u * ((u0 - 1) % kMeta), (uint32_t)((u0 - 1) / kMeta) & 1u, kWaitNs))
                return false;
            it = grab_item(p, it, lane);
            load_item(p, it < n_items ? p.items[it] : none, it < n_items, lane, cur);
        }
    } else {
        int it1 = grab_item(p, it, lane);
        const int2 rec1 = it1 < p.items_cap ? p.items[it1] : none;
        ItemPre nxt;
        load_item(p, it < n_items ? rec0 : none, it < n_items, lane, nxt);
        int2 rec2 = it1 < n_items ? rec1 : none;
        int it2 = it1 < n_items ? grab_item(p, it1, lane) : n_items;   // the item after it1
        for (; it < n_items; it = it1, it1 = it2, it2 = it2 < n_items ? grab_item(p, it2, lane) : n_items) {
            const ItemPre cur = nxt;
            load_item(p, rec2, it1 < n_items, lane, nxt);
            rec2 = it2 < n_items ? p.items[it2] : none;
            if (!publish_item(cur)) return false;
        }
    }
    if (PAIR && have_pend && !publish_joint(p, meta, mfull0, mempty0, u, lane, pend, nullptr)) return false;
    // end of stream
    const int um = u % kMeta;
    int ok = 1;
    if (lane == 0) {
        ok = mbar_wait(mempty0 + 8u * um, ((uint32_t)(u / kMeta) & 1u) ^ 1u, kWaitNs);
        if (ok) {
            meta[um].n = -1;
            __threadfence_block();
            mbar_arrive(mfull0 + 8u * um);
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// TMA warp: one stage of loads per (unit, k-block).  False after a timed-out wait;
// then the stages it filled last are waited for (bounded), so that no copy is
// still landing in shared memory when the CTA exits.
__device__ void drain_loads(const Params &p, uint32_t full0, uint32_t issued, int lane)
{
    if (lane != 0) return;
    const uint32_t S = (uint32_t)p.stages;
    for (uint32_t q = issued > S ? issued - S : 0u; q < issued; ++q)
        mbar_wait(full0 + 8u * (q % S), (q / S) & 1u, kWaitNs);
}

template <bool PAIR>
__device__ bool issue_loads(const Params &p, const UnitMeta *meta, const CUtensorMap *tmap_e,
                            const CUtensorMap *tmap_h, uint8_t *a_smem, uint8_t *b_smem, uint32_t full0,
                            uint32_t empty0, uint32_t mfull0, uint32_t mempty0, int lane)
{
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    const uint64_t evict_first = l2_policy_evict_first();
    for (int u = 0;; ++u) {
        const int um = u % kMeta;
        if (!mbar_wait(mfull0 + 8u * um, (uint32_t)(u / kMeta) & 1u, kWaitNs)) {
            drain_loads(p, full0, issued, lane);
            return false;
        }
        const UnitMeta &m = meta[um];
        const int n = m.n;
        if (n < 0) return true;
        const int nvalid = m.nvalid, g0 = m.p0;
        // lane j gathers candidate rows 4j..4j+3 (token-order table) and, for a small
        // bucket, bucket rows 4j..4j+3 while 4j < n (larger buckets: the B warps)
        const int y0 = m.tok[4 * lane] >= 0 ? m.tok[4 * lane] : p.V;
        const int y1 = m.tok[4 * lane + 1] >= 0 ? m.tok[4 * lane + 1] : p.V;
        const int y2 = m.tok[4 * lane + 2] >= 0 ? m.tok[4 * lane + 2] : p.V;
        const int y3 = m.tok[4 * lane + 3] >= 0 ? m.tok[4 * lane + 3] : p.V;
        const bool has_b = n <= kGatherRowsMax && 4 * lane < n;
        const int z0 = has_b ? m.rows[4 * lane] : 0, z1 = has_b ? m.rows[4 * lane + 1] : 0;
        const int z2 = has_b ? m.rows[4 * lane + 2] : 0, z3 = has_b ? m.rows[4 * lane + 3] : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(mempty0 + 8u * um);   // the entry is in registers now
        const bool has_a = 4 * lane < nvalid;
        const int nvalid1 = PAIR ? m.nvalid1 : 0, g1 = PAIR ? m.g1 : 0;
        const uint32_t a_tx = p.packed ? (uint32_t)(nvalid + nvalid1) * kRowBytes
                                       : (uint32_t)((nvalid + 3) / 4) * 4 * kRowBytes;
        // packed: rows [pp0, pp0 + nvalid) of the padded table, pp0 = 32*g0 (the cluster's
        // padding rows are not read; the tile rows past nvalid keep stale data, which only
        // reaches accumulator rows the epilogue skips); the run is in block pp0/128 from
        // row pp0%128 on, and continues at row 0 of the next block if it crosses the
        // block's end.  A paired unit's second chunk is a second run into tile rows 64..
        // Lanes 0-1 copy the two parts of the first run, lanes 2-3 those of the second.
        const int run = PAIR ? lane >> 1 : 0, piece = lane & 1;
        const int prow0 = (run ? g1 : g0) * kPackRows, nrows = run ? nvalid1 : nvalid;
        const int blk0 = prow0 / kPackSuper, r0 = prow0 % kPackSuper;
        const int first = min(nrows, kPackSuper - r0);
        const bool has_pk = lane < (PAIR ? 4 : 2) && nrows > 0 && (piece == 0 || nrows > first);
        const uint32_t pk_bytes = (uint32_t)(piece == 0 ? first : nrows - first) * kRowBytes;
        const uint32_t pk_dst_off =
            (run ? (uint32_t)(kTileM / 2) * kRowBytes : 0u) + (piece == 0 ? 0u : (uint32_t)first * kRowBytes);
        const uint8_t *pk_src = p.packed && has_pk ? p.packed + (size_t)(blk0 + piece) * p.num_kb * kPackBlock +
                                                         (piece == 0 ? (size_t)r0 * kRowBytes : 0)
                                                   : nullptr;
        const uint32_t tx = a_tx + (n <= kGatherRowsMax ? (uint32_t)((n + 3) / 4) * 4 * kRowBytes : 0u);
        for (int kb = 0; kb < p.num_kb; ++kb) {
            int wok = 1;
            if (lane == 0) {
                wok = mbar_wait(empty0 + 8u * stage, phase ^ 1u, kWaitNs);
                if (wok) mbar_arrive_expect_tx(full0 + 8u * stage, tx);
            }
            if (!__shfl_sync(0xffffffffu, wok, 0)) {
                drain_loads(p, full0, issued, lane);
                return false;
            }
            ++issued;
            const uint32_t bar = full0 + 8u * stage;
            const uint32_t a_dst = smem_u32(a_smem + (size_t)stage * p.a_bytes);
            if (p.packed) {
                // candidate tiles are read once per call: first out of L2, so that the
                // scatter's output rows and the hidden rows stay there
                if (has_pk)
                    bulk_copy_g2s_hint(a_dst + pk_dst_off, pk_src + (size_t)kb * kPackBlock, pk_bytes, bar,
                                       evict_first);
            } else if (has_a) {
                tma_gather4(a_dst + (uint32_t)lane * 4 * kRowBytes, tmap_e, kb * kTileK, y0, y1, y2, y3, bar);
            }
            if (has_b)
                tma_gather4(smem_u32(b_smem + (size_t)stage * p.b_bytes) + (uint32_t)lane * 4 * kRowBytes,
                            tmap_h, kb * kTileK, z0, z1, z2, z3, bar);
            if (++stage == p.stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait(int groups_in_flight)
{
    switch (groups_in_flight) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    }
}

// B warps: per (unit, k-block) the bucket's hidden rows, 64 columns each, copied
// from L2 (the whole [B, H] batch stays there) into the stage's B tile with
// 16-byte cp.async in the 128-byte swizzle; columns at or past H read as zeros.
// Thread t always copies piece t % 8 of rows t / 8, t / 8 + 16, ...  A stage is
// signalled full (one arrival per B warp) once its copies have landed and been
// fenced for the tensor cores, b_lag stages after it was filled, so that copies
// for several stages are in flight.  False after a timed-out wait (the copies
// issued are waited for and signalled before returning).
__device__ bool load_b(const Params &p, const UnitMeta *meta, uint8_t *b_smem, uint32_t full0, uint32_t empty0,
                       uint32_t mfull0, uint32_t mempty0, int bt, int lane)
{
    const int j = bt & 7, r0 = bt >> 3;
    const int S = p.stages;
    int stage = 0;
    uint32_t phase = 0, filled = 0, signalled = 0;
    bool ok = true;
    auto signal_one = [&]() {
        fence_proxy_async_smem();   // this thread's copies, visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8u * (signalled % (uint32_t)S));
        ++signalled;
    };
    // every wait is lane 0's, broadcast: the warp stays converged even if a wait gives
    // up, and __syncwarp orders the other lanes after the completion lane 0 observed
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
        int w = lane == 0 ? (int)mbar_wait(bar, parity, kWaitNs) : 1;
        w = __shfl_sync(0xffffffffu, w, 0);
        __syncwarp();
        return w != 0;
    };
    for (int u = 0; ok; ++u) {
        const int um = u % kMeta;
        const uint32_t mbar = mfull0 + 8u * um, mpar = (uint32_t)(u / kMeta) & 1u;
        // The next unit may be published only once the unit before the last one is
        // consumed (with the ticketed hand-out the metadata warp claims its next item
        // then).  A unit of fewer k-blocks than the signal lag leaves stages of that
        // earlier unit unsignalled here (more than num_kb stages owed: the last unit has
        // num_kb, each with one copy group): settle those before blocking on the next
        // unit, or their MMAs, and so the publication, could never complete.  (Units of
        // more k-blocks than the lag have signalled their predecessors by now.)
        if (filled - signalled > (uint32_t)p.num_kb) {
            int ready = lane == 0 ? (int)mbar_test_wait(mbar, mpar) : 0;
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) {
                cp_async_wait(p.num_kb);   // < b_lag groups: those of the last unit
                while (filled - signalled > (uint32_t)p.num_kb) signal_one();
            }
        }
        if (!warp_wait(mbar, mpar)) {
            ok = false;
            break;
        }
        const UnitMeta &m = meta[um];
        const int n = m.n;
        if (n < 0) break;
        const bool mine = n > kGatherRowsMax;   // small buckets come with the A tile (gather4)
        int rows[kBRowsPerThread];
#pragma unroll
        for (int i = 0; i < kBRowsPerThread; ++i) {
            const int r = r0 + 16 * i;
            rows[i] = mine && r < n ? m.rows[r] : -1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(mempty0 + 8u * um);   // the rows are in registers now
        for (int kb = 0; kb < p.num_kb; ++kb) {
            if (!warp_wait(empty0 + 8u * stage, phase ^ 1u)) {
                ok = false;
                break;
            }
            if (!mine) {
                // nothing to copy: settle the stages still owed a signal, then this one
                if (signalled < filled) {
                    cp_async_wait(0);
                    while (signalled < filled) signal_one();
                }
                ++filled;
                signal_one();
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
                continue;
            }
            const uint32_t dst0 = smem_u32(b_smem + (size_t)stage * p.b_bytes);
            const int k0 = kb * kTileK + j * 8;
            const uint32_t src_bytes = k0 < p.H ? 16u : 0u;
            const int kk = k0 < p.H ? k0 : 0;
#pragma unroll
            for (int i = 0; i < kBRowsPerThread; ++i) {
                if (rows[i] >= 0) {
                    const int r = r0 + 16 * i;
                    cp_async16(dst0 + (uint32_t)(r * kRowBytes) + (uint32_t)((j ^ (r & 7)) << 4),
                               p.hidden + (size_t)rows[i] * p.H + kk, src_bytes);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            ++filled;
            // more than b_lag stages unsignalled: the oldest one's copies have landed once at
            // most b_lag groups are pending (count the gap, not the total: small buckets
            // signal their stages at once)
            if (filled - signalled > (uint32_t)p.b_lag) {
                cp_async_wait(p.b_lag);
                signal_one();
            }
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // the stages still owed a signal (normal end or not)
    cp_async_wait(0);
    while (signalled < filled) signal_one();
    return ok;
}

template <bool SCATTER, bool PAIR>
__global__ void __launch_bounds__(kThreads, 3)
    k_gather_tc(const __grid_constant__ CUtensorMap tmap_e, const __grid_constant__ CUtensorMap tmap_h,
                const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages;
    uint8_t *a_smem = smem;
    uint8_t *b_smem = smem + (size_t)S * p.a_bytes;
    // an M = 128 MMA reads kFullABytes from a stage's base: slack after the B stages
    // keeps the last stage's read inside the allocation when a_bytes is smaller
    uint8_t *tail = b_smem + (size_t)S * p.b_bytes + (kFullABytes - p.a_bytes);
    UnitMeta *meta = reinterpret_cast<UnitMeta *>(tail);
    unsigned long long *best = reinterpret_cast<unsigned long long *>(meta + kMeta);
    uint64_t *bars = reinterpret_cast<uint64_t *>(best + p.B);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 2 * kAcc + 1 + 2 * kMeta);
    __shared__ int s_last;

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x & (kWarp - 1);
    const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8u * S;
    const uint32_t tfull0 = empty0 + 8u * S, tempty0 = tfull0 + 8u * kAcc;
    const uint32_t mfull0 = tempty0 + 8u * kAcc, mempty0 = mfull0 + 8u * kMeta;
    const uint32_t drain_bar = mempty0 + 8u * kMeta;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1 + kBWarps);   // the TMA warp (with the A bytes), the B warps
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, 4);
        }
        for (int m = 0; m < kMeta; ++m) {
            mbar_init(mfull0 + 8u * m, 1);
            mbar_init(mempty0 + 8u * m, kMetaReaders);
        }
        mbar_init(drain_bar, 1);
        fence_barrier_init();
    }
    if (!SCATTER)
        for (int b = threadIdx.x; b < p.B; b += kThreads) best[b] = 0ull;
    if (warp == 0) tmem_alloc(smem_u32(tmem_holder), p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    prefetch_l2_table(p.ordering, (size_t)p.V * sizeof(int32_t));
    prefetch_l2_table(p.offsets, (size_t)(p.C + 1) * sizeof(int32_t));
    if (p.packed) prefetch_l2_table(p.poff, (size_t)(p.C + 1) * sizeof(int32_t));
    // the work items and buckets come from the top-K kernel before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t acc_cols = p.tmem_cols / (uint32_t)p.n_acc;

    if (warp == 4) {
        if (!publish_units<PAIR>(p, meta, mfull0, mempty0, lane) && lane == 0) timeout(p);
    } else if (warp == 6) {
        if (!issue_loads<PAIR>(p, meta, &tmap_e, &tmap_h, a_smem, b_smem, full0, empty0, mfull0, mempty0, lane) &&
            lane == 0)
            timeout(p);
    } else if (warp >= 7) {
        if (!load_b(p, meta, b_smem, full0, empty0, mfull0, mempty0, threadIdx.x - 7 * kWarp, lane) && lane == 0)
            timeout(p);
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
                if (!mbar_wait(tempty0 + 8u * acc, acc_phase ^ 1u, kWaitNs)) {
                    timeout(p);
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kTileM, npad);
                const uint32_t d_tmem = tmem_base + (uint32_t)acc * acc_cols;
                bool ok = true;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(full0 + 8u * stage, phase, kWaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_kmajor_desc(smem_u32(a_smem + (size_t)stage * p.a_bytes));
                    const uint64_t bd = sw128_kmajor_desc(smem_u32(b_smem + (size_t)stage * p.b_bytes));
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
                if (++acc == p.n_acc) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued has completed before the accumulators are freed
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0u, kWaitNs);
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
            if (!mbar_wait(tfull0 + 8u * acc, acc_phase, kWaitNs)) {
                if (lane == 0) timeout(p);
                break;
            }
            tc_fence_after();
            const int t = warp * kWarp + lane;
            const int tok = m.tok[t];
            // the bucket rows that belong to this candidate's chunk (both in an unpaired unit)
            const uint8_t hbit = t >= kTileM / 2 ? 2 : 1;
            const uint32_t trow = tmem_base + ((uint32_t)(warp * kWarp) << 16) + (uint32_t)acc * acc_cols;
            for (int c0 = 0; c0 < m.npad; c0 += 16) {
                uint32_t r[16];
                tmem_load_16(trow + (uint32_t)c0, r);
                tmem_wait_load();
                if constexpr (!SCATTER) {
                    // argmax: the warp's best (logit, lower id) key of each column (bucket
                    // row) over its 32 candidates, 8 columns at a time, by a reduce-scatter
                    // butterfly: at each step a lane keeps half of its columns and takes its
                    // partner's copies of them, so after three steps the four lanes 4c..4c+3
                    // hold column c's maximum over 8 lanes each, and two more exchanges
                    // complete it; lane 4c folds it into the row's shared maximum
#pragma unroll
                    for (int h8 = 0; h8 < 16; h8 += 8) {
                        unsigned long long k[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int col = c0 + h8 + j;
                            const float v = p.bf16_logits ? round_bf16(__uint_as_float(r[h8 + j]))
                                                          : __uint_as_float(r[h8 + j]);
                            k[j] = (col < n && tok >= 0 && (!PAIR || (m.half[col] & hbit))) ? argmax_key(v, tok) : 0ull;
                        }
#pragma unroll
                        for (int h = 4, o = 16; h >= 1; h >>= 1, o >>= 1) {
                            const bool up = (lane & o) != 0;
#pragma unroll
                            for (int i = 0; i < h; ++i) {
                                const unsigned long long send = up ? k[i] : k[i + h];
                                const unsigned long long keep = up ? k[i + h] : k[i];
                                const unsigned long long recv = __shfl_xor_sync(0xffffffffu, send, o);
                                k[i] = keep > recv ? keep : recv;
                            }
                        }
#pragma unroll
                        for (int o = 2; o >= 1; o >>= 1) {
                            const unsigned long long other = __shfl_xor_sync(0xffffffffu, k[0], o);
                            k[0] = k[0] > other ? k[0] : other;
                        }
                        const int col = c0 + h8 + (((lane >> 4) & 1) << 2 | ((lane >> 3) & 1) << 1 | ((lane >> 2) & 1));
                        if (!(lane & 3) && col < n && k[0]) atomicMax(best + m.rows[col], k[0]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = c0 + j;
                        if (col >= n) break;
                        if (tok < 0 || (PAIR && !(m.half[col] & hbit))) continue;
                        const float v = p.bf16_logits ? round_bf16(__uint_as_float(r[j])) : __uint_as_float(r[j]);
                        const int row = m.rows[col];
                        if (p.sparse_width) {
                            const int rank = m.ranks[col];
                            if (rank >= 0) {
                                const size_t o = (size_t)row * p.sparse_width + (size_t)rank * p.S +
                                                 (size_t)(m.local0 + t);
                                p.out_logits[o] = v;
                                if (p.out_ids) p.out_ids[o] = tok;
                            }
                        } else {
                            p.out_logits[(size_t)row * p.V + tok] = v;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty0 + 8u * acc);
                mbar_arrive(mempty0 + 8u * um);
            }
            if (++acc == p.n_acc) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
    if constexpr (!SCATTER) {
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

size_t smem_bytes(const Params &p, int stages)
{
    return 1024 + (size_t)stages * (p.a_bytes + p.b_bytes) + (kFullABytes - p.a_bytes) +
           kMeta * sizeof(UnitMeta) + (size_t)p.B * 8 + (size_t)(2 * stages + 2 * kAcc + 1 + 2 * kMeta) * 8 + 16;
}

}  // namespace

namespace {

// Whether `n` CTAs of `kfn` with `smem` bytes of dynamic shared memory fit on one SM
// (shared memory with the per-block reservation, threads, registers), from the
// device's and the kernel's attributes (cached per kernel, device, size and count).
// The runtime's occupancy query answers one CTA here where two run side by side, so
// the fit is worked out directly; the launch asks for the largest shared-memory
// carveout so that the driver places them all.  Were the answer ever wrong, the grid
// would run in more waves: slower, still correct (the caller keeps n CTAs' TMEM
// within the SM's, so no allocation waits on a CTA that is not running).
bool ctas_fit(const void *kfn, size_t smem, int n)
{
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, size_t, int>, bool> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const auto key = std::make_tuple(kfn, dev, smem, n);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int smem_sm = 0, resv = 0, regs_sm = 0, thr_sm = 0;
    cudaFuncAttributes fa{};
    bool fit = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
               cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
               cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) == cudaSuccess &&
               cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) == cudaSuccess &&
               cudaFuncGetAttributes(&fa, kfn) == cudaSuccess;
    fit = fit && fa.numRegs > 0 &&
          (size_t)n * (smem + fa.sharedSizeBytes + (size_t)resv) <= (size_t)smem_sm && n * kThreads <= thr_sm &&
          (long long)n * kThreads * fa.numRegs <= (long long)regs_sm &&
          cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = fit;
    return fit;
}

}  // namespace

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
    p.sparse_width = g.sparse_width;
    p.bf16_logits = g.bf16_logits;
    p.out_ids = g.out_ids;
    p.topk = g.topk;
    p.K = g.K;
    p.B = g.B;
    p.H = g.H;
    p.V = g.V;
    p.S = g.S;
    p.W = g.W;
    p.C = g.C;
    p.chunk = g.chunk;
    if (p.chunk < 1 || p.chunk > kTileM) return cudaErrorInvalidValue;
    p.num_kb = (g.H + kTileK - 1) / kTileK;
    if (g.packed) {
        if (p.chunk % kPackRows != 0) return cudaErrorInvalidValue;
        p.packed = g.packed;
        p.poff = reinterpret_cast<const int32_t *>(
            g.packed + packed_poff_offset(g.V, g.H, g.C, g.packed_clusters, g.offsets != nullptr));
    }
    p.nmax = std::min(kMaxN, (g.B + 15) & ~15);
    // at most two (row, cluster) pairs per centroid: buckets are small, and units of at
    // most 32 rows let three CTAs share an SM (a rare larger bucket takes more units)
    if ((long long)g.B * g.K <= 2LL * g.C) p.nmax = std::min(p.nmax, 32);
    // the A stage holds the chunk: 32, 64 or 128 rows
    const int a_rows = p.chunk <= 32 ? 32 : p.chunk <= 64 ? 64 : kTileM;
    // With 128-row tiles and the packed table, two chunks of at most 64 candidates may
    // share a unit (not for the sparse pair, whose column blocks follow one cluster per
    // unit).  Pairing is compiled into its own kernel and chosen only where clusters
    // average at most 64 positions: with larger clusters short chunks are rare, and the
    // pairing's per-item work and registers measured ~2% slower on 128-position clusters.
    const bool pair = g.packed && a_rows == kTileM && !g.sparse_width && 2LL * g.V <= (long long)kTileM * g.C;
    p.handout = (long long)g.B * g.K >= 4LL * g.C ? 1 : 0;
    p.a_bytes = (uint32_t)a_rows * kRowBytes;
    p.b_bytes = (uint32_t)p.nmax * kRowBytes;
    uint32_t cols = 32;
    // Argmax calls with units of 64 bucket rows gathered from the token-order table run
    // three CTAs per SM with two accumulators (and two stages) each: its four-row gathers
    // keep each CTA's pipeline short of the HBM rate, so more CTAs count for more than a
    // deeper pipeline (measured on GB300 per call: shared-centroid workload B=256 166.7
    // against 184.0 us, uniform clusters B=256 216.1 against 279.2 us).  Not on the packed
    // table, whose block copies fill two CTAs' pipelines (137 against 126 us), nor for the
    // scatter, whose stores need the four accumulators' overlap (249.9 against 241.0 us).
    p.n_acc = (!g.packed && p.nmax == kMaxN && !scatter) ? 2 : kAcc;
    const int min_stages = p.n_acc == 2 ? 2 : 3;
    while (cols < (uint32_t)p.n_acc * (uint32_t)p.nmax) cols <<= 1;
    p.tmem_cols = cols;
    auto kernel = [&]() {
        if (scatter) return pair ? k_gather_tc<true, true> : k_gather_tc<true, false>;
        return pair ? k_gather_tc<false, true> : k_gather_tc<false, false>;
    }();
    const void *kfn = (const void *)kernel;
    auto fit_stages = [&](size_t budget) {
        int st = kMaxStages;
        while (st > 2 && smem_bytes(p, st) > budget) --st;
        return st;
    };
    // Two or three CTAs per SM where they fit (their accumulators within the SM's TMEM,
    // at least three stages each in their share of the shared memory): each CTA's
    // single-thread MMA issue, TMA issue and barrier round trips cost a few hundred ns
    // per k-block, so more pipelines per SM let short chunks and small H reach the HBM
    // rate and keep SMs busy through the last round of units.
    //
    // The last round of units decides the end: when few CTAs are left with a unit each,
    // each runs at its own pipeline's pace and HBM idles (at uniform B=16, ~459 units
    // over 456 CTAs, three units ran alone for ~9 us).  With uniform clusters, one item
    // per selected cluster and small buckets, the unit count is the number of distinct
    // selected clusters, expected C(1 - (1 - K/C)^B) for independent rows; where three
    // CTAs per SM would leave a thin last round and two would not, two run (measured on
    // GB300: B=16 53.1 vs 55.3 us, B=20 57.7 vs 61.7 us per call; B=12, 24 and 64, where
    // three leave a full last round, 47.1, 64.6 and 98.6 against 51.7, 68.3 and 101.5 us
    // with two).  A misprediction (rows that share clusters) costs only speed.
    int max_per_sm = 3;
    if (!p.handout && g.offsets == nullptr && (long long)g.V <= (long long)p.chunk * g.C && p.nmax >= g.B) {
        const double units = g.C * (1.0 - std::pow(1.0 - (double)g.K / g.C, (double)g.B));
        auto thin_tail = [&](int n) {
            const double rounds = units / ((double)n * sm_count());
            const double frac = rounds - std::floor(rounds + 0.05);
            return rounds >= 0.95 && frac > -0.05 && frac < 1.0 / 3.0;
        };
        if (thin_tail(3) && !thin_tail(2)) max_per_sm = 2;
    }
    int per_sm = 1;
    int stages = fit_stages(220 * 1024);
    for (int n = max_per_sm; n >= 2; --n) {
        if ((uint32_t)n * p.tmem_cols > kSmTmemCols) continue;
        const int st = fit_stages((size_t)(220 / n) * 1024);
        if (st >= min_stages && ctas_fit(kfn, smem_bytes(p, st), n)) {
            per_sm = n;
            stages = st;
            break;
        }
    }
    p.stages = stages;
    alignas(64) CUtensorMap map_e;
    // the token-order map is encoded either way (unused with the packed table)
    if (!encode_rows(&map_e, g.embed, g.H, g.V, g.ld, 1)) return cudaErrorInvalidValue;
    alignas(64) CUtensorMap map_h;
    if (!encode_rows(&map_h, g.hidden, g.H, g.B, g.H, 1)) return cudaErrorInvalidValue;
    p.hidden = g.hidden;
    p.b_lag = std::min(kBLag, p.stages - 2);
    if (p.b_lag < 0) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(p, stages);
    cudaError_t e = allow_smem(kfn, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(per_sm * sm_count()));
    return launch_dependent(kernel, grid, dim3(kThreads), smem, s, map_e, map_h, p);
}

// ---------------------------------------------------------------------------
// Packing the embedding table
// ---------------------------------------------------------------------------
namespace {

// Groups of 32 rows a table of n clusters needs (exact for uniform clusters).
size_t packed_groups_bound(int V, int C, int n, bool explicit_offsets)
{
    if (!explicit_offsets) {
        const long long S = V / C;
        return (size_t)n * (size_t)((S + kPackRows - 1) / kPackRows);
    }
    return (size_t)(((long long)V + (long long)(kPackRows - 1) * n + kPackRows - 1) / kPackRows);
}

// Padded cluster offsets, one CTA: poff[c] = sum over c' < c of roundup(size(c'), 32).
// Offsets whose padded total exceeds the buffer's bound (overlapping clusters) are
// an error: every cluster is then recorded as empty, so no later read or write
// leaves the buffer.
__global__ void __launch_bounds__(1024) k_pack_offsets(const int32_t *offsets, int V, int S, int C, int c0,
                                                       int c1, long long bound_rows, int32_t *poff, uint32_t *ctrl)
{
    __shared__ long long warp_tot[32];
    const int per = (C + (int)blockDim.x - 1) / (int)blockDim.x;
    const int cb = min(C, (int)threadIdx.x * per), ce = min(C, cb + per);
    long long local = 0;
    for (int c = cb; c < ce; ++c) {
        int lo = 0, hi = 0;
        cluster_range(offsets, V, S, c, &lo, &hi, ctrl ? ctrl + kCtrlError : nullptr);
        if (c >= c0 && c < c1) local += (hi - lo + kPackRows - 1) / kPackRows * kPackRows;
    }
    // exclusive scan of `local` over the block
    const int lane = threadIdx.x & (kWarp - 1), w = threadIdx.x / kWarp;
    const int nw = (int)blockDim.x / kWarp;
    long long incl = local;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == kWarp - 1) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
        long long t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const bool bad = warp_tot[nw - 1] > bound_rows;
    if (bad && threadIdx.x == 0 && ctrl) atomicOr(ctrl + kCtrlError, MTP_DEVERR_OFFSETS);
    long long run = bad ? 0 : incl - local + (w > 0 ? warp_tot[w - 1] : 0);
    for (int c = cb; c < ce; ++c) {
        poff[c] = (int32_t)run;
        if (bad || c < c0 || c >= c1) continue;   // other shards' clusters count as empty
        int lo = 0, hi = 0;
        cluster_range(offsets, V, S, c, &lo, &hi, nullptr);
        run += (hi - lo + kPackRows - 1) / kPackRows * kPackRows;
    }
    if (threadIdx.x == blockDim.x - 1) poff[C] = bad ? 0 : (int32_t)warp_tot[nw - 1];
}

// One CTA of 256 threads per 32-row group g and k-block kb (4 KB of the 16 KB
// block of super-group g/4): thread = (row, piece).
__global__ void __launch_bounds__(256) k_pack_tiles(const uint16_t *__restrict__ embed, long long ld,
                                                    const int32_t *__restrict__ ordering,
                                                    const int32_t *__restrict__ offsets, int V, int H, int S, int C,
                                                    int num_kb, const int32_t *__restrict__ poff,
                                                    uint8_t *__restrict__ packed, uint32_t *ctrl)
{
    __shared__ int row_tok[kPackRows];
    const int r = threadIdx.x >> 3, j = threadIdx.x & 7;
    const long long groups = __ldg(poff + C) / kPackRows;
    const long long total = groups * num_kb;
    for (long long blk = blockIdx.x; blk < total; blk += gridDim.x) {
        const long long g = blk / num_kb;
        const int kb = (int)(blk - g * num_kb);
        __syncthreads();   // the previous block's row_tok is consumed
        if (j == 0) {
            // the cluster holding padded position 32g + r: the last c with poff[c] <= pp
            const int pp = (int)(g * kPackRows) + r;
            int a = 0, b = C;   // poff[a] <= pp < poff[b] holds for the answer a
            while (b - a > 1) {
                const int mid = (a + b) >> 1;
                if (__ldg(poff + mid) <= pp) a = mid;
                else b = mid;
            }
            int lo = 0, hi = 0;
            cluster_range(offsets, V, S, a, &lo, &hi, nullptr);
            const int local = pp - __ldg(poff + a);
            int tok = -1;
            if (local < hi - lo) {
                tok = __ldg(ordering + lo + local);
                if ((unsigned)tok >= (unsigned)V) {
                    if (ctrl) atomicOr(ctrl + kCtrlError, MTP_DEVERR_TOKEN_RANGE);
                    tok = -1;
                }
            }
            row_tok[r] = tok;
        }
        __syncthreads();
        const int tok = row_tok[r];
        const int k0 = kb * kTileK + j * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tok >= 0 && k0 < H) v = ld_stream16(embed + (long long)tok * ld + k0);
        const size_t sub = ((size_t)(g / 4) * num_kb + kb) * kPackBlock + (size_t)(g % 4) * kPackRows * kRowBytes;
        uint8_t *dst = packed + sub + (size_t)r * kRowBytes + (size_t)((j ^ (r & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = v;
    }
}

}  // namespace

size_t packed_poff_offset(int V, int H, int C, int n, bool explicit_offsets)
{
    const size_t num_kb = (size_t)((H + kTileK - 1) / kTileK);
    const size_t supers = (packed_groups_bound(V, C, n, explicit_offsets) + 3) / 4;
    return supers * num_kb * kPackBlock;   // a multiple of 16 KB: poff stays 256-byte aligned
}

size_t packed_table_bytes(int V, int H, int C, int n, bool explicit_offsets)
{
    return packed_poff_offset(V, H, C, n, explicit_offsets) + (size_t)(C + 1) * sizeof(int32_t);
}

cudaError_t launch_pack_embeddings(const uint16_t *embed, long long ld, const int32_t *ordering,
                                   const int32_t *offsets, int V, int H, int C, int c0, int c1, uint8_t *packed,
                                   uint32_t *ctrl, cudaStream_t s)
{
    const int S = offsets ? 0 : V / C;
    const int n = c1 - c0;
    int32_t *poff = reinterpret_cast<int32_t *>(packed + packed_poff_offset(V, H, C, n, offsets != nullptr));
    const long long bound_rows = (long long)packed_groups_bound(V, C, n, offsets != nullptr) * kPackRows;
    k_pack_offsets<<<1, 1024, 0, s>>>(offsets, V, S, C, c0, c1, bound_rows, poff, ctrl);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int num_kb = (H + kTileK - 1) / kTileK;
    const long long total = (long long)packed_groups_bound(V, C, n, offsets != nullptr) * num_kb;
    const long long grid = std::min<long long>(total, (long long)sm_count() * 8);
    k_pack_tiles<<<(int)std::max<long long>(1, grid), 256, 0, s>>>(embed, ld, ordering, offsets, V, H, S, C,
                                                                     num_kb, poff, packed, ctrl);
    return cudaGetLastError();
}

}  // namespace mtp
