"""The cluster-sharded head across processes, against the oracle.

Two processes on one GPU each hold half of the clusters of the H=256 draft head
at Gemma scale (V=262144, C=2048, K=32).  Each computes its shard's argmax keys
with the library (mtp_masked_topk_keys), the shards exchange them with one max
all-reduce over gloo (combine_keys, the B x 8-byte exchange step that replaces
the page's all-gather of the lm_head in Gemma4MTP._get_full_lm_head_weight), and
each decodes the result (sharded_topk_tokens).  Both ranks must return the
oracle's token ids on rows whose margins are clear, and its max logits within
the tolerance.  The kernels of the two processes never wait on each other: the
exchange runs on the host between the calls.
"""
import os
import socket
import sys

import numpy as np
import pytest

from centroid_masked_sparse_gb300 import synth
from oracle import oracle
from tests import helpers

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NAME = "draft256"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, batches, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=2)
    try:
        torch.cuda.set_device(0)
        import centroid_masked_sparse_gb300 as m
        from centroid_masked_sparse_gb300 import synth as sy
        w = sy.WORKLOADS[NAME]
        t = sy.make_tables(NAME)
        full = m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets, w.top_k)
        half = w.centroids // 2
        shard = m.MaskedHead(full.centroid_w, full.embed_w, full.token_ordering, w.top_k, full.cluster_offsets,
                             vocab_size=w.vocab, cluster_range=(0, half) if rank == 0 else (half, w.centroids))
        outs = []
        for hid in batches:
            h = torch.from_numpy(hid.view(np.int16)).cuda().view(torch.bfloat16)
            tok, mx = m.sharded_topk_tokens(shard, h)
            torch.cuda.synchronize()
            outs.append((tok.cpu().numpy(), mx.cpu().numpy(), m.mtp_read_device_error(shard.workspace(len(hid)))))
        q.put((rank, outs))
    finally:
        dist.destroy_process_group()


def test_two_process_sharded_head_matches_the_oracle():
    import torch.multiprocessing as mp
    t = helpers.tables(NAME)
    oh = oracle.Head.from_tables(t, synth.WORKLOADS[NAME].top_k)
    batches, refs = [], []
    for B, row0 in ((8, 4100), (64, 4200)):   # the direct and the tensor-core gather per shard (H=256)
        hidden, ref, _ = helpers.clean_batch(NAME, oh, B, row0=row0)
        batches.append(hidden)
        refs.append(ref)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, batches, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=600) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    for rank in (0, 1):
        for (tok, mx, err), ref in zip(res[rank], refs):
            assert err == 0
            np.testing.assert_array_equal(tok, ref["tokens"], err_msg=f"rank {rank}")
            helpers.assert_close(mx, ref["max_logit"], f"rank {rank} max logit")
    # the two ranks agree bit for bit
    for a, b in zip(res[0], res[1]):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
