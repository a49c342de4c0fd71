"""Centroid-masked sparse LM head for GB300 (sm_103a).

Thin Python face of the C ABI in include/mtp_head.h: each function here has
the name of the C entry point it calls, turns torch tensors into device
pointers and the current stream into a ``cudaStream_t``, allocates outputs the
caller did not pass, and raises ``MtpError`` on a non-OK status.  Every step of
the head runs in the library's CUDA kernels; there is no other code path.

The head is Gemma4MTPMaskedEmbedder of "Add Gemma4 MTP speculative decoding
with centroids masking" (vLLM, gemma4_mtp.py): ``mtp_masked_topk_tokens`` is
get_top_tokens, ``mtp_masked_scatter_logits`` is forward,
``mtp_centroid_scores`` is the centroid Linear + topk of _select_and_score,
and ``mtp_dense_lm_head`` is the dense comparator (compute_logits without the
masked embedder, no softcapping).
"""
from __future__ import annotations

import ctypes

from ._lib import (KERNEL_IDS, MTP_DEVERR_OFFSETS, MTP_DEVERR_TIMEOUT, MTP_DEVERR_TOKEN_RANGE, MTP_MAX_BATCH,
                   MtpError, MtpHeadDesc, check, lib)

__all__ = ["MaskedHead", "MtpError", "CapturedCalls", "MTP_FINISH_ARGMAX", "MTP_FINISH_SCATTER", "MTP_FINISH_PAIR",
           "MTP_FLAG_FILL_FINFO_MIN", "MTP_FLAG_BF16_SCORES", "MTP_FLAG_BF16_LOGITS", "MTP_FLAG_HOST_HIDDEN", "mtp_workspace_bytes", "mtp_centroid_scores",
           "mtp_masked_topk_tokens", "mtp_masked_scatter_logits", "mtp_select_and_score", "mtp_dense_lm_head",
           "mtp_read_device_error", "mtp_profile_events", "mtp_packed_embeddings_bytes", "mtp_pack_embeddings", "mtp_gather_plan", "mtp_force_gather", "mtp_wait_test", "GATHER_KINDS",
           "mtp_masked_topk_keys", "mtp_decode_keys", "combine_keys", "sharded_topk_tokens",
           "MTP_DEVERR_TOKEN_RANGE",
           "MTP_DEVERR_OFFSETS", "MTP_DEVERR_TIMEOUT", "lib"]


def _torch():
    import torch
    return torch


def _stream_ptr(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class MaskedHead:
    """The head's device tables and their C descriptor.

    centroid_w       bf16 [C, H] contiguous
    embed_w          bf16 [>= V, ld] with unit inner stride (row stride ld >= H)
    token_ordering   int32 [V]: ordered position -> token id
    cluster_offsets  int32 [C + 1] or None (uniform clusters of V / C)
    cluster_range    (begin, end): the clusters this GPU owns when the head is sharded
                     over GPUs by cluster, or None for all of them
    flags            MTP_FLAG_* options: the reference-fidelity readings (0: fp32 scores and
                     logits, -inf), and MTP_FLAG_HOST_HIDDEN (hidden states may be pinned
                     CPU tensors, staged into the workspace by the call itself)
    softcap          the dense head's final logit softcap, cap * tanh(logit / cap) (0: none)
    """

    def __init__(self, centroid_w, embed_w, token_ordering, top_k, cluster_offsets=None,
                 vocab_size=None, embed_packed=None, cluster_range=None, flags=0, softcap=0.0):
        torch = _torch()
        if centroid_w is not None:
            assert centroid_w.dtype == torch.bfloat16 and centroid_w.is_contiguous()
        assert embed_w.dtype == torch.bfloat16 and embed_w.stride(1) == 1
        if token_ordering is not None:
            assert token_ordering.dtype == torch.int32 and token_ordering.is_contiguous()
        if cluster_offsets is not None:
            assert cluster_offsets.dtype == torch.int32 and cluster_offsets.is_contiguous()
        self.centroid_w = centroid_w
        self.embed_w = embed_w
        self.token_ordering = token_ordering
        self.cluster_offsets = cluster_offsets
        self.device = embed_w.device
        V = int(vocab_size if vocab_size is not None else token_ordering.shape[0])
        H = int(embed_w.shape[1]) if centroid_w is None else int(centroid_w.shape[1])
        C = 0 if centroid_w is None else int(centroid_w.shape[0])
        self.vocab_size, self.hidden_size, self.num_centroids, self.top_k = V, H, C, int(top_k)
        self.desc = MtpHeadDesc(
            vocab_size=V, hidden_size=H, num_centroids=C, top_k=int(top_k),
            device=self.device.index or 0, flags=int(flags),
            centroid_w=None if centroid_w is None else centroid_w.data_ptr(),
            embed_w=embed_w.data_ptr(), ld_embed=int(embed_w.stride(0)),
            token_ordering=None if token_ordering is None else token_ordering.data_ptr(),
            cluster_offsets=None if cluster_offsets is None else cluster_offsets.data_ptr(),
            embed_packed=None,
            cluster_begin=0 if cluster_range is None else int(cluster_range[0]),
            cluster_end=0 if cluster_range is None else int(cluster_range[1]),
            final_logit_softcap=float(softcap))
        self.cluster_range = cluster_range
        self.embed_packed = None
        self._ws = None
        if embed_packed is not None:
            self.use_packed_table(embed_packed)

    def use_packed_table(self, packed=None, stream=None):
        """Attach the packed embedding table (built here with mtp_pack_embeddings when
        not given); calls then read candidate rows as contiguous tensor-core tiles."""
        torch = _torch()
        if packed is None:
            n = mtp_packed_embeddings_bytes(self)
            packed = torch.empty(n, dtype=torch.uint8, device=self.device)
            mtp_pack_embeddings(self, packed, stream=stream)
        assert packed.dtype == torch.uint8 and packed.is_contiguous()
        self.embed_packed = packed
        self.desc.embed_packed = packed.data_ptr()
        return packed

    def with_flags(self, flags):
        """A head over the same device tables (and packed table) with other flags."""
        h = MaskedHead(self.centroid_w, self.embed_w, self.token_ordering, self.top_k,
                       self.cluster_offsets, self.vocab_size, cluster_range=self.cluster_range,
                       flags=flags, softcap=self.desc.final_logit_softcap)
        if self.embed_packed is not None:
            h.use_packed_table(self.embed_packed)
        return h

    def drop_packed_table(self):
        self.embed_packed = None
        self.desc.embed_packed = None

    @classmethod
    def from_host(cls, centroid_w, embed_w, token_ordering, cluster_offsets, top_k,
                  device="cuda", vocab_size=None):
        """Copy host numpy tables (bf16 as uint16 bit patterns) to the device."""
        torch = _torch()
        import numpy as np

        def bf16(a):
            if a is None:
                return None
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(
                torch.bfloat16)

        def i32(a):
            return None if a is None else torch.from_numpy(
                np.ascontiguousarray(a, dtype=np.int32)).to(device)

        return cls(bf16(centroid_w), bf16(embed_w), i32(token_ordering), top_k,
                   i32(cluster_offsets), vocab_size)

    def workspace(self, batch):
        """A cached workspace big enough for `batch` rows (grown on demand)."""
        torch = _torch()
        need = mtp_workspace_bytes(self, max(1, batch))
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws


def mtp_workspace_bytes(head: MaskedHead, max_batch: int) -> int:
    return int(lib().mtp_workspace_bytes(ctypes.byref(head.desc), int(max_batch)))


def _hidden_ok(head, hidden):
    """Batch rows of `hidden`: on the head's GPU, or (MTP_FLAG_HOST_HIDDEN) a pinned CPU
    tensor, which the library checks again and stages into the workspace."""
    torch = _torch()
    assert hidden.dtype == torch.bfloat16 and hidden.is_contiguous() and hidden.dim() == 2
    assert hidden.shape[1] == head.hidden_size
    if hidden.device != head.device:
        assert head.desc.flags & MTP_FLAG_HOST_HIDDEN and hidden.device.type == "cpu" and hidden.is_pinned(), \
            "hidden must be on the head's device, or a pinned CPU tensor with MTP_FLAG_HOST_HIDDEN"
    return int(hidden.shape[0])


def _out_ok(head, *outs):
    """Output arrays the device can write: on the head's GPU or pinned CPU tensors."""
    for t in outs:
        if t is not None and t.device != head.device:
            assert t.device.type == "cpu" and t.is_pinned(), \
                "outputs must be on the head's device or pinned CPU tensors"


def mtp_centroid_scores(head, hidden, scores=None, topk_idx=None, with_topk=True, stream=None):
    """(scores fp32 [B, C], topk int32 [B, K] sorted by (score desc, index asc) or None)."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    if scores is None:
        scores = torch.empty(B, head.num_centroids, dtype=torch.float32, device=head.device)
    if with_topk and topk_idx is None:
        topk_idx = torch.empty(B, head.top_k, dtype=torch.int32, device=head.device)
    check(lib().mtp_centroid_scores(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(scores),
                                    _ptr(topk_idx), _stream_ptr(stream, head.device)),
          "mtp_centroid_scores")
    return scores, topk_idx


def mtp_masked_topk_tokens(head, hidden, out_tokens=None, out_max=None, workspace=None,
                           with_max=True, stream=None):
    """(token ids int32 [B], max logit fp32 [B] or None): the sparse argmax."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    if out_tokens is None:
        out_tokens = torch.empty(B, dtype=torch.int32, device=head.device)
    if with_max and out_max is None:
        out_max = torch.empty(B, dtype=torch.float32, device=head.device)
    _out_ok(head, out_tokens, out_max)
    ws = workspace if workspace is not None else head.workspace(B)
    check(lib().mtp_masked_topk_tokens(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(out_tokens),
                                       _ptr(out_max), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream_ptr(stream, head.device)),
          "mtp_masked_topk_tokens")
    return out_tokens, out_max


def mtp_masked_scatter_logits(head, hidden, out=None, workspace=None, stream=None):
    """fp32 [B, V]: candidates' logits, -inf elsewhere."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    if out is None:
        out = torch.empty(B, head.vocab_size, dtype=torch.float32, device=head.device)
    _out_ok(head, out)
    ws = workspace if workspace is not None else head.workspace(B)
    check(lib().mtp_masked_scatter_logits(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(out),
                                          _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream_ptr(stream, head.device)),
          "mtp_masked_scatter_logits")
    return out


def mtp_select_and_score(head, hidden, out_logits=None, out_ids=None, with_ids=True, workspace=None,
                         stream=None):
    """(logits fp32 [B, K*S], token ids int32 [B, K*S] or None): _select_and_score's pair."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    width = head.top_k * (head.vocab_size // max(1, head.num_centroids))
    if out_logits is None:
        out_logits = torch.empty(B, width, dtype=torch.float32, device=head.device)
    if with_ids and out_ids is None:
        out_ids = torch.empty(B, width, dtype=torch.int32, device=head.device)
    _out_ok(head, out_logits, out_ids)
    ws = workspace if workspace is not None else head.workspace(B)
    check(lib().mtp_select_and_score(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(out_logits),
                                     _ptr(out_ids), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream_ptr(stream, head.device)), "mtp_select_and_score")
    return out_logits, out_ids


def mtp_dense_lm_head(head, hidden, out_logits=None, out_tokens=None, out_max=None,
                      want_logits=True, want_tokens=False, workspace=None, stream=None):
    """(logits fp32 [B, V] or None, token ids int32 [B] or None, max fp32 [B] or None)."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    if want_logits and out_logits is None:
        out_logits = torch.empty(B, head.vocab_size, dtype=torch.float32, device=head.device)
    if want_tokens and out_tokens is None:
        out_tokens = torch.empty(B, dtype=torch.int32, device=head.device)
        if out_max is None:
            out_max = torch.empty(B, dtype=torch.float32, device=head.device)
    _out_ok(head, out_logits, out_tokens, out_max)
    ws = None
    if out_tokens is not None or head.desc.flags & MTP_FLAG_HOST_HIDDEN:
        ws = workspace if workspace is not None else head.workspace(B)
    check(lib().mtp_dense_lm_head(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(out_logits),
                                  _ptr(out_tokens), _ptr(out_max), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream_ptr(stream, head.device)),
          "mtp_dense_lm_head")
    return out_logits, out_tokens, out_max


def mtp_packed_embeddings_bytes(head) -> int:
    return int(lib().mtp_packed_embeddings_bytes(ctypes.byref(head.desc)))


def mtp_pack_embeddings(head, out, workspace=None, stream=None):
    """Fill `out` (uint8, mtp_packed_embeddings_bytes) with the packed embedding table."""
    check(lib().mtp_pack_embeddings(ctypes.byref(head.desc), _ptr(out), out.numel(), _ptr(workspace),
                                    _stream_ptr(stream, head.device)), "mtp_pack_embeddings")
    return out


GATHER_KINDS = {0: "cuda_core", 1: "tensor_core", 2: "cuda_core_direct", 3: "fused"}


def mtp_gather_plan(head, batch: int) -> str:
    """'fused', 'cuda_core_direct', 'tensor_core' or 'cuda_core': the gather kernel a
    masked call (argmax or scatter finish) of this batch runs."""
    r = int(lib().mtp_gather_plan(ctypes.byref(head.desc), int(batch)))
    if r < 0:
        check(r, "mtp_gather_plan")
    return GATHER_KINDS[r]


def mtp_force_gather(kind):
    """Testing and profiling aid: run gather `kind` (a name of GATHER_KINDS, or None for
    the library's own choice) in every masked call of this process."""
    code = -1 if kind is None else {v: k for k, v in GATHER_KINDS.items()}[kind]
    check(lib().mtp_force_gather(code), "mtp_force_gather")


def mtp_wait_test(limit_ns: int = 0, stall: bool = False):
    """Testing aid: the pipelined gather's wait limit (0 = the default 2 s) and its stall."""
    check(lib().mtp_wait_test(int(limit_ns), 1 if stall else 0), "mtp_wait_test")


MTP_FINISH_ARGMAX, MTP_FINISH_SCATTER, MTP_FINISH_PAIR = 0, 1, 2
MTP_FLAG_FILL_FINFO_MIN, MTP_FLAG_BF16_SCORES, MTP_FLAG_BF16_LOGITS, MTP_FLAG_HOST_HIDDEN = 1, 2, 4, 8


class CapturedCalls:
    """The sparse argmax (or scatter) recorded as one CUDA graph per batch size.

    Like the fixed-size graphs the proposer keeps for get_top_tokens: each call copies
    the batch into a static input (zero-initialised, so padding rows are finite),
    replays the graph of the smallest captured size >= B and returns views of the
    first B outputs.  Batches above the largest size run the eager call.  Outputs
    are overwritten by the next call; all graphs share one workspace and run on the
    stream they were captured on (the current stream at construction by default).
    """

    def __init__(self, head, sizes=(1, 2, 4, 8, 16, 32, 64), finish="argmax", stream=None):
        torch = _torch()
        self.head, self.finish = head, finish
        self.sizes = sorted(int(b) for b in sizes)
        self.stream = stream if stream is not None else torch.cuda.current_stream(head.device)
        if self.stream.cuda_stream == 0:
            raise ValueError("graph capture needs a created stream, not the legacy default stream")
        top = self.sizes[-1]
        dev = head.device
        self.hidden = torch.zeros(top, head.hidden_size, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(mtp_workspace_bytes(head, top), dtype=torch.uint8, device=dev)
        if finish == "argmax":
            self.out0 = torch.empty(top, dtype=torch.int32, device=dev)
            self.out1 = torch.empty(top, dtype=torch.float32, device=dev)
            code = MTP_FINISH_ARGMAX
        elif finish == "scatter":
            self.out0 = torch.empty(top, head.vocab_size, dtype=torch.float32, device=dev)
            self.out1 = None
            code = MTP_FINISH_SCATTER
        elif finish == "pair":
            width = head.top_k * (head.vocab_size // max(1, head.num_centroids))
            self.out0 = torch.empty(top, width, dtype=torch.float32, device=dev)
            self.out1 = torch.empty(top, width, dtype=torch.int32, device=dev)
            code = MTP_FINISH_PAIR
        else:
            raise ValueError(finish)
        self.graphs = {}
        try:
            for b in self.sizes:
                h = ctypes.c_void_p()
                check(lib().mtp_graph_capture(ctypes.byref(head.desc), code, _ptr(self.hidden), b,
                                              _ptr(self.out0), _ptr(self.out1), _ptr(self.ws),
                                              self.ws.numel(), ctypes.c_void_p(self.stream.cuda_stream),
                                              ctypes.byref(h)), "mtp_graph_capture")
                self.graphs[b] = h
        except Exception:
            self.close()
            raise

    def size_for(self, batch):
        for b in self.sizes:
            if b >= batch:
                return b
        return None

    def replay(self, batch):
        """Replay for a batch already written into self.hidden[:batch] (no copy)."""
        size = self.size_for(batch)
        if size is None:
            raise ValueError(f"batch {batch} is above the largest captured size {self.sizes[-1]}")
        check(lib().mtp_graph_launch(self.graphs[size], ctypes.c_void_p(self.stream.cuda_stream)),
              "mtp_graph_launch")
        if self.finish in ("argmax", "pair"):
            return self.out0[:batch], self.out1[:batch]
        return self.out0[:batch]

    def __call__(self, hidden):
        B = _hidden_ok(self.head, hidden)
        size = self.size_for(B)
        with _torch().cuda.stream(self.stream):
            if size is None:   # above the largest graph: the eager call
                if self.finish == "argmax":
                    return mtp_masked_topk_tokens(self.head, hidden)
                if self.finish == "pair":
                    return mtp_select_and_score(self.head, hidden)
                return mtp_masked_scatter_logits(self.head, hidden)
            self.hidden[:B].copy_(hidden)
            check(lib().mtp_graph_launch(self.graphs[size], ctypes.c_void_p(self.stream.cuda_stream)),
                  "mtp_graph_launch")
        if self.finish in ("argmax", "pair"):
            return self.out0[:B], self.out1[:B]
        return self.out0[:B]

    def close(self):
        for h in self.graphs.values():
            lib().mtp_graph_destroy(h)
        self.graphs = {}

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass


def mtp_masked_topk_keys(head, hidden, out_keys=None, workspace=None, stream=None):
    """int64 [B]: this shard's best candidate of each row as a max-combinable key."""
    torch = _torch()
    B = _hidden_ok(head, hidden)
    if out_keys is None:
        out_keys = torch.empty(B, dtype=torch.int64, device=head.device)
    _out_ok(head, out_keys)
    ws = workspace if workspace is not None else head.workspace(B)
    check(lib().mtp_masked_topk_keys(ctypes.byref(head.desc), _ptr(hidden), B, _ptr(out_keys), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream_ptr(stream, head.device)),
          "mtp_masked_topk_keys")
    return out_keys


def mtp_decode_keys(keys, out_tokens=None, out_max=None, with_max=True, stream=None):
    """(token ids int32 [B], max logit fp32 [B] or None) from combined keys."""
    torch = _torch()
    B = int(keys.shape[0])
    assert keys.dtype == torch.int64 and keys.is_contiguous()
    if out_tokens is None:
        out_tokens = torch.empty(B, dtype=torch.int32, device=keys.device)
    if with_max and out_max is None:
        out_max = torch.empty(B, dtype=torch.float32, device=keys.device)
    check(lib().mtp_decode_keys(_ptr(keys), B, _ptr(out_tokens), _ptr(out_max),
                                _stream_ptr(stream, keys.device)), "mtp_decode_keys")
    return out_tokens, out_max


def combine_keys(keys, group=None):
    """The shards' exchange step: an elementwise max of the int64 keys over the ranks of
    `group` (in place).  Nothing to do without an initialised process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1):
        return keys
    if keys.is_cuda and dist.get_backend(group) == "gloo":
        # gloo reduces host tensors: the B x 8 bytes go through host memory
        host = keys.cpu()
        dist.all_reduce(host, op=dist.ReduceOp.MAX, group=group)
        keys.copy_(host)
    else:
        dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)
    return keys


def sharded_topk_tokens(head, hidden, group=None, workspace=None, stream=None):
    """The sparse argmax of a cluster-sharded head: each rank's keys over its clusters,
    one max all-reduce of B x 8 bytes, then the decode (same result on every rank)."""
    keys = mtp_masked_topk_keys(head, hidden, workspace=workspace, stream=stream)
    combine_keys(keys, group)
    return mtp_decode_keys(keys, stream=stream)


def mtp_read_device_error(workspace, stream=None) -> int:
    """The device error word of the last call that used `workspace` (synchronises the stream)."""
    torch = _torch()
    word = ctypes.c_uint32(0)
    st = torch.cuda.current_stream(workspace.device) if stream is None else stream
    check(lib().mtp_read_device_error(_ptr(workspace), ctypes.byref(word),
                                      ctypes.c_void_p(st.cuda_stream)), "mtp_read_device_error")
    st.synchronize()
    return int(word.value)


def mtp_profile_events(kernel: str, start=None, stop=None) -> None:
    """Record torch.cuda.Event pair around one kernel of every following call (None clears)."""
    check(lib().mtp_profile_events(KERNEL_IDS[kernel],
                                   None if start is None else ctypes.c_void_p(start.cuda_event),
                                   None if stop is None else ctypes.c_void_p(stop.cuda_event)),
          "mtp_profile_events")
