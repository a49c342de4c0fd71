"""The multi-replica path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Rows are independent, so N GPUs run N replicas with no collective on the data
path; what the ranks share is the timing: a barrier on both sides of the timed
loop, the slowest rank's time (all-reduce max) and the whole-job rate.  The
reference arm runs on rank 0 only.  No GPU is used."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, _ = bench.dist_setup()
        bench.barrier(got_ws)
        # each rank's call time differs; the job is as slow as its slowest rank
        call_ms = 0.1 + 0.05 * rank
        slowest = bench.max_over_ranks(call_ms, got_ws)
        value = bench.job_tokens_per_s(got_ws, 64, slowest)
        bench.barrier(got_ws)
        q.put((got_rank, got_ws, slowest, value, bench.rank_row0(got_rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_barrier_and_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    # both ranks see the slowest time (0.15 ms) and the same whole-job rate: 2 x 64 rows / 0.15 ms
    for r in res:
        assert r[2] == pytest.approx(0.15)
        assert r[3] == pytest.approx(2 * 64 / 0.15e-3)
    # the replicas draw disjoint hidden rows
    assert res[0][4] != res[1][4]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "3"]
    r1 = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r0 = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_starts_its_own_ranks():
    """`bench.py --gpus 2` outside a launcher starts two ranks itself (torch.distributed.run
    on 127.0.0.1): the reference arm's line, printed by rank 0 alone, reports both ranks,
    with the same `config` object as the library's arm."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    sys.path.insert(0, ROOT)
    import bench
    from centroid_masked_sparse_gb300 import synth
    args = bench.parse_args(["--workload", "tiny", "--gpus", "2"])
    assert line["config"] == bench.run_config(args, synth.WORKLOADS["tiny"], 1, 2)


def _key(logit, token):
    """A key in the order the library's keys follow: larger logit, then lower token id,
    as a signed 64-bit integer (used here only to feed the exchange step)."""
    import struct
    bits = struct.unpack("<I", struct.pack("<f", logit))[0]
    ordv = bits | 0x80000000 if bits < 0x80000000 else (~bits) & 0xFFFFFFFF
    u = (ordv << 32) | (0xFFFFFFFF - token)
    u ^= 1 << 63
    return u - (1 << 64) if u >= 1 << 63 else u


def _combine_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=ws)
    try:
        from centroid_masked_sparse_gb300 import combine_keys
        # row 0: rank 1 has the larger logit; row 1: equal logits, rank 0 has the lower id;
        # row 2: only rank 0 has a candidate (rank 1 reports "none"); row 3: negative logits
        mine = {0: [_key(1.5, 10), _key(2.0, 7), _key(0.25, 3), _key(-3.0, 5)],
                1: [_key(2.5, 99), _key(2.0, 8), -(1 << 63), _key(-2.0, 6)]}[rank]
        keys = torch.tensor(mine, dtype=torch.int64)
        combine_keys(keys)
        q.put((rank, keys.tolist()))
    finally:
        dist.destroy_process_group()


def test_sharded_argmax_exchange_is_a_max_all_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_combine_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=5) for _ in range(2))
    want = [_key(2.5, 99), _key(2.0, 7), _key(0.25, 3), _key(-2.0, 6)]
    assert res[0] == want and res[1] == want


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The bench's `roofline.traffic` comes from a committed ncu summary only while the
    summary's source hash matches the kernel file, and summaries of the token-order table
    are looked up under `_token` (a packed-table summary never stands in for them)."""
    import bench
    csrc = tmp_path / "centroid_masked_sparse_gb300" / "csrc"
    prof = tmp_path / "profiles"
    csrc.mkdir(parents=True)
    prof.mkdir()
    (csrc / "gather_tc.cu").write_text("// kernel source\n")
    sha = bench.file_sha(str(csrc / "gather_tc.cu"))
    (prof / "gather_tc_shared_b256.md").write_text(f"dram_bytes_per_launch: 1000\nsource_sha256_16: {sha}\n")
    (prof / "gather_tc_shared_token_b256.md").write_text(f"dram_bytes_per_launch: 2000\nsource_sha256_16: {sha}\n")
    (prof / "gather_tc_uniform_b64.md").write_text("dram_bytes_per_launch: 3000\nsource_sha256_16: 0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("gather_tc", "shared", 256) == 1000.0
    assert bench.profiled_traffic("gather_tc", "shared", 256, "token") == 2000.0
    assert bench.profiled_traffic("gather_tc", "uniform", 64) is None          # stale hash
    assert bench.profiled_traffic("gather_tc", "uniform", 64, "token") is None # no summary
    assert bench.profiled_traffic(None, "shared", 256) is None
