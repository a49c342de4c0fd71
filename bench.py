"""Benchmark of the centroid-masked sparse LM head on one GB300 (or N replicas).

Default workload: Gemma-scale uniform clusters, V=262144 as 2048 clusters of
128 tokens, H=1536, K=32 (4096 candidates a row), batch 64, sparse-argmax
finish (mtp_masked_topk_tokens).  A step is one call of the whole head on one
batch of synthetic hidden states, with the tables already resident in HBM.
L2 is flushed before every timed call, outside the events: a 256 MB write, then a
512 MB read, so the written lines are evicted (and written back) before the
call starts instead of inside it.

Printed (rank 0, one JSON line): draft tokens/s over all ranks, µs per call,
the gather-score kernel's roofline against the measured HBM copy bandwidth,
the oracle's CPU throughput on a bounded sample, an end-to-end figure through
the C ABI with host buffers (H2D of the hidden states and D2H of the tokens
inside the timed region), SM clocks sampled during the timed loop, and a
sweep over batch 1..64 plus the other finishes and cluster layouts.

--impl reference times the oracle (the plain fp64 CPU implementation) on the
host cores instead, on the same workload and metric.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked-head draft tokens/s"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20
EVICT_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file, workload, batch, layout="packed"):
    """DRAM bytes per launch from a committed ncu summary, if it still matches the kernel source
    (summaries of the token-order table carry `_token` after the workload's name)."""
    if kernel_file is None:
        return None
    suffix = "_token" if layout == "token" else ""
    prof = os.path.join(ROOT, "profiles", f"{kernel_file}_{workload}{suffix}_b{batch}.md")
    src = os.path.join(ROOT, "centroid_masked_sparse_gb300", "csrc", f"{kernel_file}.cu")
    try:
        text = open(prof).read()
    except OSError:
        return None
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", text)
    m_s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_s or m_s.group(1) != file_sha(src):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running."""

    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid=None):
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) != len(self.FIELDS):
                continue
            try:
                ts = time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
                rows.append((ts, float(p[1]), float(p[2]), p[5], p[6], p[7], p[8]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        note = "samples inside the timed loop"
        if not inside and rows:
            rows.sort(key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))
            inside = rows[:3]
            note = "nearest samples to a timed loop shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "none"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_row0(rank):
    """First hidden-row index of a rank's batches: every replica draws its own rows."""
    return rank * 100000


def job_tokens_per_s(ws, batch_per_rank, slowest_call_ms):
    """Whole-job rate: the rows all ranks processed per call, over the slowest rank's time."""
    return ws * batch_per_rank / (slowest_call_ms * 1e-3)


def max_over_ranks(x, ws, device=None):
    """The maximum of a float over all ranks (the slowest rank sets the time)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workload description and byte model
# ---------------------------------------------------------------------------

def cluster_sizes(t):
    w = t.workload
    if t.cluster_offsets is not None:
        return np.diff(t.cluster_offsets.astype(np.int64))
    return np.full(w.centroids, w.vocab // w.centroids, dtype=np.int64)


def byte_model(t, sel, B, scatter):
    """Algorithmic bytes of one call: each distinct candidate row once, each table once.

    call:   B*H*2 (hidden) + C*H*2 (centroid table) + U*(2H + 4) (distinct candidate rows and
            their token_ordering entries) + (C+1)*4 (offsets, if any) + output
    gather: U*(2H + 4) + B*H*2 + output of the gather kernel
    output: B*8 (argmax keys / tokens) or B*V*4 (full-vocabulary rows)."""
    w = t.workload
    H, C, V = w.hidden, w.centroids, w.vocab
    uniq = np.unique(sel)
    usz = int(cluster_sizes(t)[uniq].sum())
    cand = int(sum(cluster_sizes(t)[sel[b]].sum() for b in range(B)))
    out = B * V * 4 if scatter else B * 8
    offs = (C + 1) * 4 if t.cluster_offsets is not None else 0
    call = B * H * 2 + C * H * 2 + usz * (2 * H + 4) + offs + out
    gather = usz * (2 * H + 4) + B * H * 2 + (cand * 4 if scatter else B * 8)
    return dict(call=call, gather=gather, unique_clusters=int(uniq.size), unique_tokens=usz,
                candidates_per_row=cand / B)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Timer:
    def __init__(self, torch, m, device):
        self.torch, self.m, self.device = torch, m, device
        self.flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.evict = torch.ones(EVICT_BYTES // 4, dtype=torch.float32, device=device)

    def flush_l2(self):
        """Write 256 MB (the flush), then read 512 MB: L2 ends up holding clean lines of
        a buffer the call never touches, so no write-back of the flush lands in the call."""
        self.flush.zero_()
        self.evict.sum()

    def before_call(self, flush):
        """Outside the timed events: the L2 flush, or (warm figure) a ~100 us spin kernel,
        so that in both cases the GPU is busy while the host enqueues the call and the
        call's launches are queued before it starts (no host launch gap inside it)."""
        if flush:
            self.flush_l2()
        else:
            self.torch.cuda._sleep(200000)

    def events(self, n):
        torch = self.torch
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:          # create the driver events now (torch creates them on first record)
            e.record()
        return evs

    def run(self, fn, steps, warmup, kernel=None, ws=1, extra_kernels=(), flush=True):
        """Per-step device times (ms) of fn(i) and of library kernels (events the library
        records around each launch on the call's stream).  flush=False: L2 keeps what the
        previous call left (the warm figure)."""
        torch, m = self.torch, self.m
        for i in range(warmup):
            self.before_call(flush)
            fn(i)
        names = ([kernel] if kernel else []) + [k for k in extra_kernels if k != kernel]
        call_ev = self.events(2 * steps)
        kev = {k: self.events(2 * steps) for k in names}
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        # no garbage collection inside the loop: a collection that stalls the host long
        # enough to drain the launch queue would leave the GPU idle inside a timed call
        gc.collect()
        gc.disable()
        try:
            t0 = time.time()
            for i in range(steps):
                self.before_call(flush)
                for k in names:
                    m.mtp_profile_events(k, kev[k][2 * i], kev[k][2 * i + 1])
                call_ev[2 * i].record()
                fn(i)
                call_ev[2 * i + 1].record()
            torch.cuda.synchronize()
        finally:
            gc.enable()
        barrier(ws)
        torch.cuda.synchronize()
        t1 = time.time()
        for k in names:
            m.mtp_profile_events(k, None, None)
        call = [call_ev[2 * i].elapsed_time(call_ev[2 * i + 1]) for i in range(steps)]
        per = {k: [kev[k][2 * i].elapsed_time(kev[k][2 * i + 1]) for i in range(steps)] for k in names}
        if names:
            self.last_breakdown = {k: float(np.mean(v)) for k, v in per.items()}
        kern = per[kernel] if kernel else None
        return call, kern, t0, t1


def make_batches(synth, t, name, B, n, row0):
    w = synth.WORKLOADS[name]
    return [synth.hidden_batch(w, B, None, t.prototypes, row0=row0 + j * B) for j in range(n)]


def measure_masked(ctx, t, dh, name, B, steps, warmup, scatter=False, rot=4, row0=0):
    torch, m, synth, timer = ctx["torch"], ctx["m"], ctx["synth"], ctx["timer"]
    hb = make_batches(synth, t, name, B, rot, row0)
    hs = [torch.from_numpy(h.view(np.int16)).to(ctx["device"]).view(torch.bfloat16) for h in hb]
    ws = dh.workspace(B)
    if scatter:
        out = torch.empty(B, t.workload.vocab, dtype=torch.float32, device=ctx["device"])
        fn = lambda i: m.mtp_masked_scatter_logits(dh, hs[i % rot], out=out, workspace=ws)  # noqa: E731
    else:
        tok = torch.empty(B, dtype=torch.int32, device=ctx["device"])
        mx = torch.empty(B, dtype=torch.float32, device=ctx["device"])
        fn = lambda i: m.mtp_masked_topk_tokens(dh, hs[i % rot], out_tokens=tok, out_max=mx,  # noqa: E731
                                                workspace=ws)
    # the headline: whole calls, no library events between the kernels (events recorded
    # between launches would also stop the dependent-launch overlap)
    call, _, t0, t1 = timer.run(fn, steps, warmup, ws=ctx["ws"])
    # secondary: the same calls back to back without the flush (the batch's rows and the
    # tables' hot lines may still be in L2 from the previous call; at small batches the
    # whole working set fits)
    warm, _, _, _ = timer.run(fn, max(20, steps // 4), 2, ws=ctx["ws"], flush=False)
    # the per-kernel breakdown, in a separate shorter loop with the library's events (the
    # fused small-batch kernel selects the top-K itself: no top-K launch then)
    fused = m.mtp_gather_plan(dh, B) == "fused"
    extra = ("projection",) + (() if fused else ("topk",)) + (("fill",) if scatter else ())
    _, kern, _, _ = timer.run(fn, max(20, steps // 4), 2, kernel="gather_score", ws=ctx["ws"],
                              extra_kernels=extra)
    breakdown = {k: round(v * 1e3, 2) for k, v in timer.last_breakdown.items()}
    # every timed call must have run clean (no device-side error or timeout)
    dev_err = m.mtp_read_device_error(ws)
    # byte model from the library's own selection of each rotated batch
    models = []
    for h in hs:
        _, topk = m.mtp_centroid_scores(dh, h)
        models.append(byte_model(t, topk.cpu().numpy(), B, scatter))
    bm = {k: float(np.mean([d[k] for d in models])) for k in models[0]}
    call_ms = float(np.mean(call))
    kern_ms = float(np.mean(kern))
    return dict(call_ms=call_ms, kernel_ms=kern_ms, t0=t0, t1=t1, bytes=bm,
                launches_per_call=(2 if fused else 3) + (1 if scatter else 0), kernels_us=breakdown,
                max_call_us=round(float(np.max(call)) * 1e3, 2),
                warm_l2_us_per_call=round(float(np.mean(warm)) * 1e3, 2),
                median_call_us=round(float(np.median(call)) * 1e3, 2), device_error=dev_err)


def measure_graph(ctx, t, dh, name, B, steps, warmup, rot=4, row0=0):
    """µs per call replaying a CUDA graph of the call (the batch copied into the graph's
    static input inside the timed region), on a side stream: the legacy stream cannot be
    captured.  Medians: the loops are short, and one host stall would dominate a mean."""
    torch, m, synth, timer = ctx["torch"], ctx["m"], ctx["synth"], ctx["timer"]
    hb = make_batches(synth, t, name, B, rot, row0)
    hs = [torch.from_numpy(h.view(np.int16)).to(ctx["device"]).view(torch.bfloat16) for h in hb]
    gs = torch.cuda.Stream(device=ctx["device"])
    gs.wait_stream(torch.cuda.current_stream(ctx["device"]))
    with torch.cuda.stream(gs):
        g = m.CapturedCalls(dh, sizes=(B,))
        try:
            call, _, _, _ = timer.run(lambda i: g(hs[i % rot]), steps, warmup, ws=ctx["ws"])
            # replay alone: the producer of the hidden states wrote them into the static input
            g.hidden[:B].copy_(hs[0])
            bare, _, _, _ = timer.run(lambda i: g.replay(B), steps, warmup, ws=ctx["ws"])
            err = m.mtp_read_device_error(g.ws, stream=gs)
        finally:
            gs.synchronize()
            g.close()
    torch.cuda.current_stream(ctx["device"]).wait_stream(gs)
    return float(np.median(call)), float(np.median(bare)), err


def measure_pair(ctx, t, dh, name, B, steps, warmup, rot=4, row0=0):
    """µs per call of the sparse pair (mtp_select_and_score) and its gather kernel's µs."""
    torch, m, synth, timer = ctx["torch"], ctx["m"], ctx["synth"], ctx["timer"]
    hb = make_batches(synth, t, name, B, rot, row0)
    hs = [torch.from_numpy(h.view(np.int16)).to(ctx["device"]).view(torch.bfloat16) for h in hb]
    ws = dh.workspace(B)
    width = t.workload.top_k * (t.workload.vocab // t.workload.centroids)
    lg = torch.empty(B, width, dtype=torch.float32, device=ctx["device"])
    ids = torch.empty(B, width, dtype=torch.int32, device=ctx["device"])
    fn = lambda i: m.mtp_select_and_score(dh, hs[i % rot], out_logits=lg, out_ids=ids,  # noqa: E731
                                          workspace=ws)
    call, _, _, _ = timer.run(fn, steps, warmup, ws=ctx["ws"])
    _, kern, _, _ = timer.run(fn, max(20, steps // 4), 2, kernel="gather_score", ws=ctx["ws"])
    return dict(call_ms=float(np.mean(call)), kernel_ms=float(np.mean(kern)),
                device_error=m.mtp_read_device_error(ws), out_bytes=B * width * 8)


def measure_dense(ctx, t, dh, B, steps, warmup):
    torch, m, synth, timer = ctx["torch"], ctx["m"], ctx["synth"], ctx["timer"]
    h = torch.from_numpy(synth.hidden_batch("scatter", B).view(np.int16)).to(ctx["device"]).view(
        torch.bfloat16)
    out = torch.empty(B, t.workload.vocab, dtype=torch.float32, device=ctx["device"])
    fn = lambda i: m.mtp_dense_lm_head(dh, h, out_logits=out)  # noqa: E731
    call, _, _, _ = timer.run(fn, steps, warmup, ws=ctx["ws"])
    _, kern, _, _ = timer.run(fn, max(10, steps // 2), 2, kernel="dense", ws=ctx["ws"])
    w = t.workload
    byts = w.vocab * w.hidden * 2 + B * w.hidden * 2 + B * w.vocab * 4
    ms = float(np.mean(kern))
    return dict(call_ms=float(np.mean(call)), kernel_ms=ms, bytes=byts,
                flops=2.0 * B * w.vocab * w.hidden)


def measure_e2e(ctx, t, dh, name, B, steps, warmup, copy_engine=False):
    """Through the C ABI with host buffers, inside the timed region every step: the
    step's hidden states go from pinned host memory to the GPU and its token ids and max
    logits come back to pinned host memory.  Default: the library's host-input path
    (MTP_FLAG_HOST_HIDDEN: the call's own staging kernel reads the pinned batch over the
    host link; the gather's last CTA writes the results into pinned memory).
    copy_engine: a cudaMemcpyAsync in, the call on device buffers, a cudaMemcpyAsync out."""
    torch, m, synth = ctx["torch"], ctx["m"], ctx["synth"]
    hb = make_batches(synth, t, name, B, 4, 20000)
    host_in = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).pin_memory() for h in hb]
    # token ids and max logits side by side in one buffer
    host_out = torch.empty(2 * B, dtype=torch.int32).pin_memory()
    if copy_engine:
        dev_in = torch.empty(B, t.workload.hidden, dtype=torch.bfloat16, device=ctx["device"])
        dev_out = torch.empty(2 * B, dtype=torch.int32, device=ctx["device"])
        tok, mx = dev_out[:B], dev_out[B:].view(torch.float32)
        ws = dh.workspace(B)

        def fn(i):
            dev_in.copy_(host_in[i % 4], non_blocking=True)
            m.mtp_masked_topk_tokens(dh, dev_in, out_tokens=tok, out_max=mx, workspace=ws)
            host_out.copy_(dev_out, non_blocking=True)
    else:
        hh = dh.with_flags(dh.desc.flags | m.MTP_FLAG_HOST_HIDDEN)
        tok, mx = host_out[:B], host_out[B:].view(torch.float32)
        ws = hh.workspace(B)

        def fn(i):
            m.mtp_masked_topk_tokens(hh, host_in[i % 4], out_tokens=tok, out_max=mx, workspace=ws)

    call, _, _, _ = ctx["timer"].run(fn, steps, warmup, ws=ctx["ws"])
    return float(np.mean(call)), B * t.workload.hidden * 2, B * 8


def cpu_baseline(t, name, B, budget_s=10.0, threads=None):
    """The oracle as it stands, on the host cores, on a bounded sample of the workload."""
    from centroid_masked_sparse_gb300 import synth
    from oracle import oracle
    threads = threads or os.cpu_count() or 1
    head = oracle.Head.from_tables(t)
    hidden = synth.hidden_batch(synth.WORKLOADS[name], B, None, t.prototypes)
    rows = 0
    t0 = time.time()
    passes = 0
    while True:
        oracle.masked_topk_tokens(head, hidden, threads=threads)
        rows += B
        passes += 1
        if time.time() - t0 >= budget_s:
            break
    dt = time.time() - t0
    return dict(value=rows / dt, unit=UNIT, cores=threads, kind="oracle",
                sample=f"{passes} passes over one {B}-row batch of the '{name}' workload "
                       f"(sparse argmax, fp64 plain C, rows spread over {threads} threads)",
                us_per_call=dt / passes * 1e6)


def run_config(args, w, B, ws):
    """The `config` object of the JSON line: the same for the library's arm and the
    reference arm on the same workload."""
    return {"workload": workload_label(w, B), "finish": "sparse argmax",
            "embedding_layout": ("packed tiles (built once at load, outside the timing)"
                                 if args.layout == "packed" else "token order"),
            "batch_per_gpu": B, "parallelism": "replicas" if ws > 1 else "single",
            "l2": "flushed before every timed call, outside the events: 256 MB written, "
                  "then 512 MB read so the written lines are evicted before the call"}


def workload_label(w, B):
    layout = "lognormal clusters" if w.variable_clusters else f"{w.centroids}x{w.vocab // w.centroids} clusters"
    return (f"{w.name}: V={w.vocab} ({layout}), H={w.hidden}, C={w.centroids}, K={w.top_k}, B={B}")


def gpu_main(args):
    ws, rank, local = dist_setup()
    import torch
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import centroid_masked_sparse_gb300 as m
    from centroid_masked_sparse_gb300 import build, synth
    build.build()
    ctx = dict(torch=torch, m=m, synth=synth, device=device, ws=ws, timer=Timer(torch, m, device))
    hbm, hbm_src = peaks()

    name = args.workload
    w = synth.WORKLOADS[name]
    B = args.batch or w.batch
    t = synth.make_tables(name)
    dh = m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets,
                                w.top_k, device=device)
    dh_packed = dh.use_packed_table() if args.layout == "packed" else None
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:  # noqa: BLE001
        uuid = None
    if args.finish != "argmax":
        # profiling aid: one finish only, a short line with its timing (not the headline)
        if args.finish == "dense":
            r = measure_dense(ctx, t, dh, B, args.steps, args.warmup)
            print(json.dumps({"finish": "dense", "workload": workload_label(w, B),
                              "us_per_call": round(r["call_ms"] * 1e3, 2),
                              "kernel_us": round(r["kernel_ms"] * 1e3, 2),
                              "gbs": round(r["bytes"] / (r["kernel_ms"] * 1e-3) / 1e9, 1)}))
        else:
            r = measure_masked(ctx, t, dh, name, B, args.steps, args.warmup, scatter=True)
            print(json.dumps({"finish": "scatter", "workload": workload_label(w, B),
                              "us_per_call": round(r["call_ms"] * 1e3, 2),
                              "kernels_us": r["kernels_us"], "device_error": r["device_error"]}))
        return
    sampler = ClockSampler(uuid) if rank == 0 else None
    res = measure_masked(ctx, t, dh, name, B, args.steps, args.warmup, row0=rank_row0(rank))
    clocks = sampler.stop(res["t0"], res["t1"]) if sampler else None
    call_ms = max_over_ranks(res["call_ms"], ws, device)
    value = job_tokens_per_s(ws, B, call_ms)
    kern_s = res["kernel_ms"] * 1e-3
    achieved = res["bytes"]["gather"] / kern_s / 1e9
    plan = m.mtp_gather_plan(dh, B)
    kfile, kname = {"tensor_core": ("gather_tc", "k_gather_tc"), "fused": ("select_gather", "k_select_gather"),
                    "cuda_core_direct": (None, "k_gather_direct")}.get(plan, ("score", "k_gather_score"))
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                "peak": hbm, "peak_source": f"{hbm_src} HBM copy GB/s", "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": profiled_traffic(kfile, name, B, args.layout),
                "algorithmic_bytes": int(res["bytes"]["gather"]),
                "kernel_us": round(res["kernel_ms"] * 1e3, 2)}
    call_gbs = res["bytes"]["call"] / (res["call_ms"] * 1e-3) / 1e9
    out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(call_ms, 5),
           "us_per_call": round(call_ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": run_config(args, w, B, ws),
           "call_roofline": {"achieved": round(call_gbs, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(call_gbs / hbm, 4),
                             "algorithmic_bytes": int(res["bytes"]["call"]),
                             "unique_clusters": res["bytes"]["unique_clusters"]},
           "roofline": roofline,
           "kernels_us": res["kernels_us"],
           "max_call_us": res["max_call_us"], "median_call_us": res["median_call_us"],
           "warm_l2_us_per_call": res["warm_l2_us_per_call"],
           "device_error": res["device_error"],
           "gpu_launches": res["launches_per_call"] * args.steps,
           "clocks": clocks}

    if rank == 0 and not args.quick:
        e2e_ms, bi, bo = measure_e2e(ctx, t, dh, name, B, max(20, args.steps // 2), args.warmup)
        ce_ms, _, _ = measure_e2e(ctx, t, dh, name, B, max(20, args.steps // 2), args.warmup,
                                  copy_engine=True)
        out["e2e"] = {"value": round(B / (e2e_ms * 1e-3), 1), "unit": UNIT,
                      "us_per_call": round(e2e_ms * 1e3, 2),
                      "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                      "path": "pinned host batch read by the call's staging kernel "
                              "(MTP_FLAG_HOST_HIDDEN); token ids and max logits written by the "
                              "kernel into pinned host memory",
                      "copy_engine_us_per_call": round(ce_ms * 1e3, 2)}
        sweep = {}
        for b in (w.batches or (B,)):
            r = measure_masked(ctx, t, dh, name, b, max(20, args.steps // 4), args.warmup,
                               row0=40000 + b)
            ach = r["bytes"]["gather"] / (r["kernel_ms"] * 1e-3) / 1e9
            cg = r["bytes"]["call"] / (r["call_ms"] * 1e-3) / 1e9
            g_ms, g_bare_ms, g_err = measure_graph(ctx, t, dh, name, b, max(20, args.steps // 4),
                                                   args.warmup, row0=40000 + b)
            sweep[str(b)] = {"gather_kernel": m.mtp_gather_plan(dh, b),
                             "us_per_call": round(r["call_ms"] * 1e3, 2),
                             "graph_us_per_call": round(g_ms * 1e3, 2),
                             "graph_replay_only_us": round(g_bare_ms * 1e3, 2), "graph_device_error": g_err,
                             "tokens_per_s": round(b / (r["call_ms"] * 1e-3), 1),
                             "gather_us": round(r["kernel_ms"] * 1e3, 2),
                             "gather_gbs": round(ach, 1), "gather_frac": round(ach / hbm, 4),
                             "call_gbs": round(cg, 1), "call_frac": round(cg / hbm, 4),
                             "unique_clusters": r["bytes"]["unique_clusters"],
                             "kernels_us": r["kernels_us"], "max_call_us": r["max_call_us"],
                             "warm_l2_us_per_call": r["warm_l2_us_per_call"],
                             "device_error": r["device_error"]}
        out["sweep"] = sweep
        if args.layout == "packed":
            # the same workload on the token-order table alone (no packed copy)
            dh.drop_packed_table()
            r = measure_masked(ctx, t, dh, name, B, max(20, args.steps // 4), args.warmup, row0=60000)
            out["token_order_layout"] = {"us_per_call": round(r["call_ms"] * 1e3, 2),
                                         "tokens_per_s": round(B / (r["call_ms"] * 1e-3), 1),
                                         "gather_us": round(r["kernel_ms"] * 1e3, 2),
                                         "kernels_us": r["kernels_us"]}
            dh.use_packed_table(dh_packed)
        if not args.no_extra:
            out["other_workloads"] = other_workloads(ctx, args, hbm)
        out["cpu_baseline"] = cpu_baseline(t, name, B, budget_s=args.cpu_seconds)
        one = cpu_baseline(t, name, B, budget_s=max(2.0, args.cpu_seconds / 2), threads=1)
        out["cpu_baseline"]["one_thread"] = {"value": one["value"], "unit": UNIT, "cores": 1,
                                             "us_per_call": one["us_per_call"], "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def other_workloads(ctx, args, hbm):
    """The scatter finish, variable clusters, shared centroids and the dense comparator."""
    m, synth, torch = ctx["m"], ctx["synth"], ctx["torch"]
    res = {}
    steps = max(10, args.steps // 8)
    cases = (("scatter", True, False), ("scatter", True, True), ("variable", False, False), ("shared", False, False),
             ("shared", True, False), ("uniform", False, False), ("uniform", False, True),
             ("variable", False, True), ("shared", False, True), ("shared", True, True),
             ("draft256", False, False), ("draft256", False, True))
    for name, scatter, packed in cases:
        w = synth.WORKLOADS[name]
        t = synth.make_tables(name)
        dh = m.MaskedHead.from_host(t.centroid_w, t.embed_w, t.token_ordering, t.cluster_offsets,
                                    w.top_k, device=ctx["device"])
        if packed:
            dh.use_packed_table()
        r = measure_masked(ctx, t, dh, name, w.batch, steps, args.warmup, scatter=scatter)
        cg = r["bytes"]["call"] / (r["call_ms"] * 1e-3) / 1e9
        ga = r["bytes"]["gather"] / (r["kernel_ms"] * 1e-3) / 1e9
        key = f"{name}_{'scatter' if scatter else 'argmax'}_b{w.batch}"
        if packed:
            key += "_packed_table"
        res[key] = {"workload": workload_label(w, w.batch),
                    "us_per_call": round(r["call_ms"] * 1e3, 2),
                    "tokens_per_s": round(w.batch / (r["call_ms"] * 1e-3), 1),
                    "call_gbs": round(cg, 1), "call_frac": round(cg / hbm, 4),
                    "gather_us": round(r["kernel_ms"] * 1e3, 2), "gather_gbs": round(ga, 1),
                    "gather_frac": round(ga / hbm, 4),
                    "unique_clusters": r["bytes"]["unique_clusters"],
                    "kernels_us": r["kernels_us"], "max_call_us": r["max_call_us"],
                    "device_error": r["device_error"]}
        if name == "uniform" and not scatter:
            pr = measure_pair(ctx, t, dh, name, w.batch, steps, args.warmup)
            res[f"uniform_pair_b{w.batch}" + ("_packed_table" if packed else "")] = {
                "finish": "sparse pair (logits + token ids, [B, K*S])",
                "us_per_call": round(pr["call_ms"] * 1e3, 2),
                "tokens_per_s": round(w.batch / (pr["call_ms"] * 1e-3), 1),
                "gather_us": round(pr["kernel_ms"] * 1e3, 2), "output_bytes": pr["out_bytes"],
                "device_error": pr["device_error"]}
        if name == "scatter" and not packed:
            d = measure_dense(ctx, t, dh, w.batch, steps, args.warmup)
            gbs = d["bytes"] / (d["kernel_ms"] * 1e-3) / 1e9
            res[f"dense_b{w.batch}"] = {"us_per_call": round(d["call_ms"] * 1e3, 2),
                                        "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                        "tflops": round(d["flops"] / (d["kernel_ms"] * 1e-3) / 1e12, 2)}
        del dh
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------

def reference_main(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    from centroid_masked_sparse_gb300 import synth
    from oracle import oracle
    oracle.build()
    name = args.workload
    w = synth.WORKLOADS[name]
    B = args.batch or w.batch
    t = synth.make_tables(name)
    head = oracle.Head.from_tables(t)
    threads = os.cpu_count() or 1
    batches = [synth.hidden_batch(w, B, None, t.prototypes, row0=j * B) for j in range(2)]
    for i in range(args.warmup):
        oracle.masked_topk_tokens(head, batches[i % 2][:max(1, B // 8)], threads=threads)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle.masked_topk_tokens(head, batches[i % 2], threads=threads)
        times.append(time.perf_counter() - t0)
    step_s = float(np.mean(times))
    value = B / step_s
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": run_config(args, w, B, ws),
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads,
                            "kind": "oracle",
                            "sample": f"each step: one {B}-row batch of the '{name}' workload, "
                                      f"rows spread over {threads} threads"},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="uniform")
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--quick", action="store_true", help="headline line only")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layout", default="packed", choices=["packed", "token"],
                    help="embedding table the calls read: the packed tile copy (built once, outside "
                         "the timing) or the token-order table alone")
    ap.add_argument("--finish", default="argmax", choices=["argmax", "scatter", "dense"],
                    help="profiling aid: time only this finish on the workload's tables")
    a = ap.parse_args(argv)
    a.warmup = max(3, a.warmup)
    return a


def spawn_ranks(n):
    """`--gpus N` (N > 1) outside a launcher: start N ranks of this same command line on
    this node with torch.distributed.run (one process per GPU, rendezvous on 127.0.0.1)
    and return their exit status; rank 0 prints the JSON line."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


if __name__ == "__main__":
    args = parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus))
    if args.impl == "reference":
        reference_main(args)
    else:
        gpu_main(args)
