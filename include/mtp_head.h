/*
 * mtp_head.h - C ABI of the centroid-masked sparse LM head for GB300 (sm_103a).
 *
 * The head computes, for each draft hidden state h (one row of the batch):
 *   1. centroid scores   s[c] = sum_k h[k] * Wc[c, k]                (C scores)
 *   2. top-K centroids   the K largest scores (lower index first on ties)
 *   3. candidates        the token ids owned by those centroids: centroid c
 *                        owns ordered positions [off[c], off[c+1]) and
 *                        token_ordering[p] is the token id at position p
 *   4. sparse logits     logit[t] = sum_k h[k] * E[t, k] for every candidate t
 * and finishes either with the token id of the largest sparse logit, or with
 * a full-vocabulary fp32 row holding each candidate's logit and -inf
 * elsewhere.  This is Gemma4MTPMaskedEmbedder of "Add Gemma4 MTP speculative
 * decoding with centroids masking" (vLLM, vllm/model_executor/models/
 * gemma4_mtp.py): __init__ (V/C tokens per centroid, bias-free centroid Linear
 * [C, H], token_ordering buffer [V]), _select_and_score (steps 1-4),
 * get_top_tokens (sparse argmax) and forward (full-vocabulary scatter).  The
 * dense comparator is the compute_logits fallback of Gemma4MTP (the
 * LogitsProcessor over every vocabulary row) without final softcapping.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All array pointers are DEVICE pointers on desc->device and are owned by
 *   the caller.  The library never allocates or frees device memory, never
 *   synchronises, and never reads device memory on the host, so every call is
 *   a pure sequence of kernel launches (and, for the dense head, one
 *   cudaMemsetAsync) on `stream`.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 * - bf16 arrays are raw IEEE bfloat16 bit patterns (uint16 storage).
 * - Rows are row-major.  hidden is [batch, H] with row stride H.
 * - Host-side argument checks run before anything is launched; a failed check
 *   returns its status and launches nothing.  A launch failure returns
 *   MTP_ERR_CUDA.  Problems that only the device can see (a token id outside
 *   [0, V), cluster offsets that are not ascending inside [0, V]) do not
 *   fault: the offending entry is skipped and a bit is set in the workspace's
 *   device error word (see mtp_read_device_error).
 * - A workspace serves one call at a time: concurrent calls on different
 *   streams need different workspaces.  Tables may be shared freely.
 * - A call makes desc->device current while it launches and gives the calling
 *   thread back its own current device before it returns.
 *
 * Readings of the source that this library takes (where the page is silent or
 * inconsistent): token ids are int32 (the page uses int64); scores and logits
 * are fp32 with fp32 accumulation from bf16 inputs (the page's Linear/einsum
 * produce bf16); top-K ties go to the lower centroid index; argmax ties go to
 * the lower token id; the full-vocabulary fill is -inf (the docstring of
 * forward), not the dtype's finite minimum; no final logit softcapping.
 */
#ifndef MTP_HEAD_H
#define MTP_HEAD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MTP_API __attribute__((visibility("default")))
#else
#define MTP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mtp_status {
    MTP_OK = 0,
    MTP_ERR_NULL = -1,        /* a required pointer is NULL                         */
    MTP_ERR_SHAPE = -2,       /* a size is out of range or inconsistent             */
    MTP_ERR_ALIGN = -3,       /* a pointer or row stride is not 16-byte aligned     */
    MTP_ERR_WORKSPACE = -4,   /* workspace NULL or smaller than mtp_workspace_bytes */
    MTP_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed               */
    MTP_ERR_UNSUPPORTED = -6  /* valid but outside the library's limits (see below) */
} mtp_status;

/* Limits of the library (MTP_ERR_UNSUPPORTED beyond them):
 *   H % 8 == 0 and 8 <= H <= 4096; 1 <= K <= C <= 16384; 1 <= batch <= 1024;
 *   1 <= V < 2^31; uniform clusters need V % C == 0. */
#define MTP_MAX_HIDDEN 4096
#define MTP_MAX_CENTROIDS 16384
#define MTP_MAX_BATCH 1024

/* Bits of the device error word (OR-ed together over one call). */
#define MTP_DEVERR_TOKEN_RANGE 0x1u  /* token_ordering held an id outside [0, V) */
#define MTP_DEVERR_OFFSETS 0x2u      /* cluster_offsets not ascending in [0, V]  */
#define MTP_DEVERR_TIMEOUT 0x4u      /* a bounded wait of a pipelined kernel gave
                                        up (its results are invalid; nothing hung) */

/* The head's tables.  Plain data: the struct is read on the host at each call
 * and may live anywhere on the host.
 *   vocab_size       V, number of tokens (rows of embed_w that are used)
 *   hidden_size      H, length of a hidden state, of a centroid row, of an embedding row
 *   num_centroids    C
 *   top_k            K, centroids selected per row
 *   device           CUDA ordinal that holds every buffer of the calls
 *   centroid_w       bf16 [C, H] row-major (the Linear weight layout); 16-byte aligned
 *   embed_w          bf16 [>= V, ld_embed], token-id order (the lm_head weight; rows
 *                    at or beyond V, e.g. padding, are never read); 16-byte aligned
 *   ld_embed         elements between consecutive rows of embed_w; >= H, multiple of 8
 *   token_ordering   int32 [V]: ordered position -> token id; must be a permutation of
 *                    0..V-1 (not checked; a duplicate id makes the scatter's winner
 *                    for that id unspecified)
 *   cluster_offsets  int32 [C+1] ascending, off[0] = 0, off[C] = V: centroid c owns
 *                    positions [off[c], off[c+1]); empty clusters are allowed.  NULL
 *                    means uniform clusters of V/C positions (the page's layout).
 *   embed_packed     optional packed copy of the embedding table built by
 *                    mtp_pack_embeddings (layout below), 256-byte aligned.  When set,
 *                    the masked calls that run the tensor-core gather read each chunk's
 *                    candidate rows as runs of contiguous 16 KB blocks instead of
 *                    gathering them row by row, and the library routes more calls
 *                    there (see mtp_gather_plan).  Token
 *                    ids are the same either way; logits agree within fp32 rounding
 *                    of the summation order (bit for bit when the same gather kernel
 *                    runs).  NULL: gather from embed_w (the page's layout).  It must
 *                    have been packed from this descriptor's tables; the library does
 *                    not check that.
 *   cluster_begin,   the clusters this GPU owns when the head is sharded over GPUs by
 *   cluster_end      cluster: [cluster_begin, cluster_end), 0 <= begin <= end <= C;
 *                    (0, 0) means all clusters.  The projection and top-K still run
 *                    over all C centroids (the centroid table is replicated); only
 *                    selected clusters inside the range are gathered.  The argmax
 *                    finish then gives this shard's best candidate of each row
 *                    (combine shards with mtp_masked_topk_keys, a max all-reduce and
 *                    mtp_decode_keys), the scatter finish writes only this shard's
 *                    candidates (-inf elsewhere; the elementwise max over shards is
 *                    the whole row), and a packed table holds only these clusters.
 *                    embed_w stays indexed by token id; only the rows of this
 *                    shard's tokens are read.
 *   final_logit_softcap  the dense head's final logit softcap (the page's dense path,
 *                    Gemma4MTP.compute_logits, applies final_logit_softcapping): each
 *                    dense logit becomes cap * tanh(logit / cap) before it is stored,
 *                    rounded (MTP_FLAG_BF16_LOGITS) or compared; 0 = none.  The masked
 *                    calls never apply it (the page's masked path does not).  Negative
 *                    or NaN: MTP_ERR_SHAPE. */
/* Reference-fidelity options (desc->flags; 0 = the library's default reading:
 * fp32 scores and logits, -inf fill).  The page's head runs in the model dtype,
 * bf16 ("Add Gemma4 MTP speculative decoding with centroids masking",
 * gemma4_mtp.py, Gemma4MTPMaskedEmbedder._select_and_score and forward):
 *   MTP_FLAG_FILL_FINFO_MIN  the full-vocabulary scatter fills with bf16's finite
 *                            minimum (-3.3895314e38, torch.finfo(bfloat16).min)
 *                            instead of -inf;
 *   MTP_FLAG_BF16_SCORES     the top-K selects on the centroid scores rounded to
 *                            bf16 (round to nearest even; ties then go to the
 *                            lower centroid index); the fp32 scores that
 *                            mtp_centroid_scores returns are not rounded;
 *   MTP_FLAG_BF16_LOGITS     every sparse and dense logit is rounded to bf16 before
 *                            it is stored and before the argmax (ties then go to
 *                            the lower token id); outputs stay fp32 arrays.
 * An input-placement option, not a reading of the page:
 *   MTP_FLAG_HOST_HIDDEN     `hidden` may live in pinned host memory (cudaHostAlloc,
 *                            cudaMallocHost, or cudaHostRegister'ed memory, at its
 *                            device address: the same as the host address under
 *                            unified addressing).  The call first copies the batch's
 *                            rows into its workspace with one kernel of this
 *                            library reading over the host link, then reads only
 *                            that copy; this replaces a separate host-to-device
 *                            copy ahead of the call and the wait for it.  The
 *                            pointer is checked with cudaPointerGetAttributes:
 *                            host memory the device cannot address (pageable,
 *                            unregistered) or another GPU's memory give
 *                            MTP_ERR_UNSUPPORTED and nothing is launched; device
 *                            and managed memory are accepted and copied the same
 *                            way.  The workspace grows by batch * H * 2 bytes
 *                            (mtp_workspace_bytes counts it); calls without a
 *                            workspace (mtp_centroid_scores, and the dense head
 *                            without one) return MTP_ERR_UNSUPPORTED with it.
 *                            Output arrays need no flag: any address the device
 *                            can write works, pinned host memory included.
 * Other bits: MTP_ERR_UNSUPPORTED. */
#define MTP_FLAG_FILL_FINFO_MIN 1
#define MTP_FLAG_BF16_SCORES 2
#define MTP_FLAG_BF16_LOGITS 4
#define MTP_FLAG_HOST_HIDDEN 8

typedef struct mtp_head_desc {
    int32_t vocab_size;
    int32_t hidden_size;
    int32_t num_centroids;
    int32_t top_k;
    int32_t device;
    int32_t flags;
    const void *centroid_w;
    const void *embed_w;
    int64_t ld_embed;
    const int32_t *token_ordering;
    const int32_t *cluster_offsets;
    const void *embed_packed;
    int32_t cluster_begin;
    int32_t cluster_end;
    float final_logit_softcap;
} mtp_head_desc;

/* Bytes of device workspace that the masked calls and the dense head's argmax
 * need for batches of up to max_batch rows.  Pure host arithmetic; returns 0
 * if the descriptor's sizes or max_batch are invalid.  The workspace needs no
 * initialisation: every call resets the parts it uses.  Its first 4 bytes are
 * the device error word of the last call that used it. */
MTP_API size_t mtp_workspace_bytes(const mtp_head_desc *desc, int32_t max_batch);

/* Steps 1-2 (the centroid Linear and topk of _select_and_score).
 *   hidden    bf16 [batch, H], 16-byte aligned
 *   scores    fp32 [batch, C] out: s[b, c]
 *   topk_idx  int32 [batch, K] out, or NULL: the selected centroids of each row,
 *             sorted by (score desc, index asc) like a sorted topk
 * Needs no workspace (so MTP_FLAG_HOST_HIDDEN is not accepted here). */
MTP_API mtp_status mtp_centroid_scores(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                               float *scores, int32_t *topk_idx, void *stream);

/* get_top_tokens: steps 1-4 and the sparse argmax, without a full-vocabulary row.
 *   out_tokens  int32 [batch] out: token id of the largest sparse logit of each row
 *               (lower id on exact ties); -1 if the row's selected clusters are all
 *               empty
 *   out_max     fp32 [batch] out, or NULL: that logit (-inf for a -1 row)
 *   workspace   device buffer of at least mtp_workspace_bytes(desc, batch) bytes,
 *               16-byte aligned */
MTP_API mtp_status mtp_masked_topk_tokens(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                                  int32_t *out_tokens, float *out_max,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* forward: steps 1-4 written into a full-vocabulary row.
 *   out_logits  fp32 [batch, V] out, row stride V, 16-byte aligned: the sparse
 *               logit at each candidate token id, -inf at every other id */
MTP_API mtp_status mtp_masked_scatter_logits(const mtp_head_desc *desc, const void *hidden,
                                     int32_t batch, float *out_logits,
                                     void *workspace, size_t workspace_bytes, void *stream);

/* _select_and_score: steps 1-4 returned as the sparse pair, for consumers of the
 * candidates themselves (tree drafting, sampling over the candidate set).  Uniform
 * clusters only (cluster_offsets NULL; MTP_ERR_UNSUPPORTED otherwise): with
 * S = V / C, row b holds K*S entries, the clusters in the row's selection order
 * (score desc, index asc) and inside each cluster its positions in order:
 *   out_logits  fp32 [batch, K*S] out: entry k*S + i is the logit of token
 *               token_ordering[c_k * S + i], c_k the row's k-th selected centroid
 *   out_ids     int32 [batch, K*S] out, or NULL: that token id
 * Every entry is written (no fill); with an out-of-range token id in
 * token_ordering the entries of that id are left unwritten and the device error
 * word reports MTP_DEVERR_TOKEN_RANGE.  Workspace as for mtp_masked_topk_tokens. */
MTP_API mtp_status mtp_select_and_score(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                                        float *out_logits, int32_t *out_ids, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* Dense comparator: logit[b, t] = sum_k h[b, k] * E[t, k] for every t < V.
 *   out_logits  fp32 [batch, V] out (row stride V), or NULL
 *   out_tokens  int32 [batch] out, or NULL: dense argmax, lower id on ties
 *   out_max     fp32 [batch] out, or NULL (only with out_tokens)
 *   workspace   needed only when out_tokens != NULL or with MTP_FLAG_HOST_HIDDEN
 *               (same size rule as above)
 * centroid_w, token_ordering and cluster_offsets are not read; at least one of
 * out_logits and out_tokens must be non-NULL. */
MTP_API mtp_status mtp_dense_lm_head(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                             float *out_logits, int32_t *out_tokens, float *out_max,
                             void *workspace, size_t workspace_bytes, void *stream);

/* Sparse argmax for callers that cannot allocate device memory.  The paper
 * has no counterpart of this call; it exists for callers that are handed only
 * their input and output buffers (for example a plugin or custom-operator
 * interface that passes tensors but no allocator) or that cannot afford
 * cudaMalloc's possible device-wide synchronisation, and so cannot supply the
 * workspace of mtp_masked_topk_tokens.
 *
 * Same arguments and results as mtp_masked_topk_tokens, without the
 * workspace: the call uses a scratch array of MTP_NOALLOC_SCRATCH_BYTES that
 * lives in the library's own device memory (every GPU that loads the library
 * holds it until the process exits).  It calls no allocating routine.
 *   - Sizes: accepted only if mtp_workspace_bytes(desc, batch) <=
 *     MTP_NOALLOC_SCRATCH_BYTES; larger requests return MTP_ERR_UNSUPPORTED
 *     and launch nothing.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress, with desc->device made current) and
 *     caches it; make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, and the array keeps
 *     the last call's contents (each call clears what must start at zero).
 *     Calls whose kernels overlap on the GPU (different streams without
 *     ordering between them) race on the array and give undefined results.
 *   - Checks: the same host-side checks as mtp_masked_topk_tokens run first,
 *     with the same statuses, before the size limit and the set-up.
 *   - Device reset: the cached address belongs to the device's context; after
 *     cudaDeviceReset on that device the entry point must not be used again in
 *     this process.
 *   - Errors found on the device (the device error word) go to the array's
 *     first word: read them with mtp_noalloc_read_device_error on the same
 *     device and stream after the call; the next call on the device resets it. */
#define MTP_NOALLOC_SCRATCH_BYTES (8u << 20)
MTP_API mtp_status mtp_masked_topk_tokens_noalloc(const mtp_head_desc *desc, const void *hidden,
                                                  int32_t batch, int32_t *out_tokens,
                                                  float *out_max, void *stream);

/* The device error word of the last mtp_masked_topk_tokens_noalloc call on
 * `device`, copied asynchronously into *host_word on `stream` (valid once the
 * stream has been synchronised); see mtp_read_device_error.  Allocates
 * nothing. */
MTP_API mtp_status mtp_noalloc_read_device_error(int32_t device, uint32_t *host_word, void *stream);

/* The packed embedding table: the rows of each cluster in ordered-position
 * order, cut into the operand tiles of the tensor-core gather.  This is a
 * layout of this library (the page gathers from the token-order table on every
 * call); building it is a one-time step, like loading the weights.
 *
 * Layout, with KB = ceil(H / 64) k-blocks of 64 elements:
 *   - cluster c is padded to P(c) = roundup(size(c), 32) positions; padded
 *     cluster offsets poff[c] = P(0) + ... + P(c-1); padded position q of
 *     cluster c (q < size(c)) is the embedding row of token_ordering[off[c] + q];
 *   - padded positions 128s .. 128s+127 (super-group s) and k-block kb form one
 *     16384-byte block at byte offset (s * KB + kb) * 16384: its row r (0..127)
 *     holds elements kb*64 .. kb*64+63 of padded position 128s + r (zeros for
 *     padding rows and for elements at or beyond H), with the 16-byte piece j
 *     (elements j*8 .. j*8+7) stored at r*128 + ((j XOR (r mod 8)) * 16), the
 *     128-byte swizzle the tensor cores read;
 *   - after the blocks (SG = ceil(groups / 4) super-groups, groups the bound
 *     below): int32 poff[0..C].
 * mtp_packed_embeddings_bytes gives the size for the descriptor's shapes: with
 * uniform clusters exactly n * ceil(S/32) groups of 32, with explicit cluster
 * offsets the upper bound ceil((V + 31 n) / 32) groups, n the clusters the
 * descriptor owns (cluster_end - cluster_begin, or C); 0 for an invalid
 * descriptor.  A sharded descriptor's table holds only its clusters (the others
 * count as empty in poff). */
MTP_API size_t mtp_packed_embeddings_bytes(const mtp_head_desc *desc);

/* Fill `packed` (packed_bytes >= mtp_packed_embeddings_bytes(desc), 256-byte
 * aligned, not overlapping the tables) from desc->embed_w, token_ordering and
 * cluster_offsets.  Reads V*H*2 bytes and writes the packed size; asynchronous on
 * `stream`.  Token ids outside [0, V) become zero rows and, like invalid cluster
 * offsets (clusters then count as empty), set MTP_DEVERR_TOKEN_RANGE /
 * MTP_DEVERR_OFFSETS in *workspace's error word when workspace is non-NULL
 * (16-byte aligned, at least 64 bytes; the word is not cleared first). */
MTP_API mtp_status mtp_pack_embeddings(const mtp_head_desc *desc, void *packed, size_t packed_bytes,
                                       void *workspace, void *stream);

/* The sparse argmax as per-row keys, for combining shards of a cluster-sharded
 * head (desc->cluster_begin/end) across GPUs: out_keys[b] orders this shard's
 * best candidate of row b so that the larger signed 64-bit value is the larger
 * logit, the lower token id on equal logits, and INT64_MIN means no candidate.
 * The shards' keys combine by an elementwise max (an all-reduce with MAX over
 * int64); mtp_decode_keys turns the result into token ids and logits.
 *   out_keys   int64 [batch] out
 * Workspace as for mtp_masked_topk_tokens. */
MTP_API mtp_status mtp_masked_topk_keys(const mtp_head_desc *desc, const void *hidden, int32_t batch,
                                        int64_t *out_keys, void *workspace, size_t workspace_bytes,
                                        void *stream);

/* Keys of mtp_masked_topk_keys (after any combination) -> out_tokens int32
 * [batch] (-1 for INT64_MIN) and out_max fp32 [batch] or NULL (-inf for -1). */
MTP_API mtp_status mtp_decode_keys(const int64_t *keys, int32_t batch, int32_t *out_tokens,
                                   float *out_max, void *stream);

/* CUDA graphs of the masked calls.  Gemma4Proposer._setup_centroids_cuda_graphs
 * ("Add Gemma4 MTP speculative decoding with centroids masking", vLLM
 * spec_decode/gemma4.py) records get_top_tokens at fixed batch sizes so that a
 * draft step replays one graph instead of launching its kernels one by one.
 * mtp_graph_capture does the same for one call with fixed buffers: it runs the
 * call once eagerly on `stream` (argument checks, one-time per-device setup),
 * then records it (cudaStreamBeginCapture in thread-local mode) and instantiates
 * the graph.  Every pointer (desc tables, hidden, outputs, workspace) is baked
 * in: a replay reads the buffers' contents at replay time, so the caller copies
 * each new batch into `hidden` before mtp_graph_launch.  The descriptor struct
 * itself is not kept.
 *   finish   MTP_FINISH_ARGMAX: out0 = int32 out_tokens [batch], out1 = float
 *            out_max [batch] or NULL (mtp_masked_topk_tokens);
 *            MTP_FINISH_SCATTER: out0 = float out_logits [batch, V], out1 unused
 *            (mtp_masked_scatter_logits);
 *            MTP_FINISH_PAIR: out0 = float out_logits [batch, K*S], out1 = int32
 *            out_ids [batch, K*S] or NULL (mtp_select_and_score)
 *   stream   a created stream (capture is impossible on the legacy stream: NULL
 *            returns MTP_ERR_NULL)
 *   graph    receives an opaque handle owned by the caller (mtp_graph_destroy)
 * Replays of one graph on several streams at once race on its workspace.  The
 * eager call's statuses apply; a failed capture returns MTP_ERR_CUDA and leaves
 * *graph NULL. */
#define MTP_FINISH_ARGMAX 0
#define MTP_FINISH_SCATTER 1
#define MTP_FINISH_PAIR 2
typedef struct mtp_graph mtp_graph;
MTP_API mtp_status mtp_graph_capture(const mtp_head_desc *desc, int32_t finish, const void *hidden,
                                     int32_t batch, void *out0, void *out1, void *workspace,
                                     size_t workspace_bytes, void *stream, mtp_graph **graph);
/* Enqueue one replay of the recorded call on `stream` (any stream of the graph's device). */
MTP_API mtp_status mtp_graph_launch(const mtp_graph *graph, void *stream);
/* Free the graph (NULL is a no-op).  The caller must not destroy a graph whose
 * replay is still in flight. */
MTP_API mtp_status mtp_graph_destroy(mtp_graph *graph);

/* Which gather kernel a masked argmax or scatter call with this descriptor and
 * batch runs: 3 for the fused small-batch kernel, which selects each row's top-K
 * itself right behind the projection (batches of at most 8 rows, 10 with uniform
 * clusters and H <= 1536, with K <= 1024 and
 * H > 256), else 2 for the direct CUDA-core gather (at H <= 256 up to 10 rows with a
 * packed table and 20 without, and
 * at most 12 rows where the tensor-core gather would not run), else 1 for the
 * tensor-core gather (large buckets, batch * K >= 4C; or with a packed table batch *
 * K >= C/5 for uniform clusters and >= C/4 with cluster_offsets; or batch * K >= C/4
 * at H <= 256; or >= C/16 with a packed table and H <= 256), else 0 for the pipelined
 * CUDA-core gather; a negative mtp_status for
 * an invalid descriptor or batch, or MTP_ERR_UNSUPPORTED when mtp_force_gather
 * forces a kernel that cannot run this call.  The sparse pair runs only kernels 0
 * and 1.  Host-only; for profiling and benchmarks (the calls choose by
 * themselves). */
MTP_API int32_t mtp_gather_plan(const mtp_head_desc *desc, int32_t batch);

/* Testing and profiling aid (not part of the head): make the masked argmax and
 * scatter calls (and the sparse pair) run gather kernel `kind` (the numbers of
 * mtp_gather_plan) whatever the batch; -1 restores the library's own choice.
 * Calls that the forced kernel cannot run (the fused and direct kernels do not
 * produce the sparse pair; the direct one takes at most 32 rows and
 * batch * H * 2 <= 200 KB; the fused one K <= 1024) return MTP_ERR_UNSUPPORTED
 * and launch nothing.  Results do not depend on the kernel beyond fp32 rounding
 * of the summation order.  Process-wide, not thread-safe.  Out-of-range kind:
 * MTP_ERR_SHAPE. */
MTP_API mtp_status mtp_force_gather(int32_t kind);

/* Testing aid for the bounded waits (not part of the head).  Every mbarrier wait
 * of the pipelined CUDA-core gather (kernel 0 of mtp_gather_plan) gives up after
 * a wall-clock limit, sets MTP_DEVERR_TIMEOUT in the device error word and lets
 * its CTA finish; the call's results are then invalid but nothing hangs, and the
 * next call starts clean.  limit_ns > 0 sets that limit (default 2 s; 0 restores
 * the default).  stall != 0 makes the first hidden-row buffer wait of every CTA
 * that has work wait for a barrier phase that nothing completes, before the CTA
 * has issued any copy: the wait runs out after limit_ns, and so do the waits of
 * the CTA's consumer warps, which then have nothing to consume.  Process-wide,
 * not thread-safe; a negative limit gives MTP_ERR_SHAPE. */
MTP_API mtp_status mtp_wait_test(int64_t limit_ns, int32_t stall);

/* Enqueue an asynchronous copy of the workspace's device error word (a set of
 * MTP_DEVERR_* bits, reset by each masked call) into *host_word; the value is
 * valid once `stream` has been synchronised. */
MTP_API mtp_status mtp_read_device_error(const void *workspace, uint32_t *host_word, void *stream);

/* Static English text for a status code. */
MTP_API const char *mtp_status_string(mtp_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
MTP_API int32_t mtp_version(void);

/* Profiling aid (not part of the head): while set, every call records
 * `start_event` on its stream just before launching kernel `kernel` and
 * `stop_event` just after it (events are cudaEvent_t passed as void*; NULL
 * clears).  kernel: 0 projection, 1 top-K/bucket, 2 gather-score, 3 -inf
 * fill, 4 dense head.  Process-wide, not thread-safe. */
#define MTP_KERNEL_PROJECTION 0
#define MTP_KERNEL_TOPK 1
#define MTP_KERNEL_GATHER_SCORE 2
#define MTP_KERNEL_FILL 3
#define MTP_KERNEL_DENSE 4
MTP_API mtp_status mtp_profile_events(int32_t kernel, void *start_event, void *stop_event);

#ifdef __cplusplus
}
#endif

#endif /* MTP_HEAD_H */
