"""Decode-step benchmark of libkvr on one B300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen3-4b-128k|llama3.1-8b-32k|qwen3-4b-128k-host]
                    [--step sequential|overlap|pipeline] [--layers L] [--no-extras]
                    [--e2e-calls C] [--copies R] [--kernel-launches L] [--no-cpu-baseline]

One step is one speculative decode step of one attention layer over a batch
of sequences, through kvr_speculative_step (default): page scoring, then the
top-k selection per KV head with the group-similarity correction decision,
then the sparse GQA attention over the pages each KV head uses this step.
``--step overlap`` runs kvr_speculative_step_overlap instead (the selection
on a side stream beside the reused heads' attention).  Page summaries are
built once per cache (prefill) and reported on their own.  Inputs are seeded
synthetic caches with the layer shapes of Qwen3-4B at 128K context (default)
or Llama-3.1-8B at 32K; the queries follow the AR(1) trace of the speculative
workload.  The cache, queries and state are resident in HBM before the timed
region; four copies of the cache (--copies) rotate so that no step reads
data a recent step left in L2.  Exactly K steps are timed: a CUDA graph of
min(64, K) captured steps is replayed K // 64 times, plus a graph of the
remaining steps.  Per-kernel times come from graphs of 64 back-to-back calls
of each kind, replayed until at least --kernel-launches calls have run.  The
line's "also" key holds compact records of the other HBM workload and of the
host-resident one (--no-extras drops them).  The "-host" workload keeps the
cache in page-locked host memory and recalls the selected pages every step
(kvr_speculative_step_recall).  ``--step pipeline`` runs a decode step
through --layers layers with kvr_pipeline_step instead (stand-in projection
reads between the attentions), beside the same layers stepped one call at a
time, and reports a per-layer latency breakdown.

The line's "e2e" is the same step through the public call a serving loop
makes with host buffers, kvr_speculative_step_host: every step reads its
query from pinned host memory and leaves its output there, with one step in
flight (2000 timed eager calls after 200 untimed ones, --e2e-calls); it also
reports the rate when the host waits for every step.

Prints one JSON line (rank 0).  With --impl reference the fp64 oracle is
timed instead, on the host's cores, over a bounded sample of the workload
(its speculative steps, in segments of 8 steps of the same query trace).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s and selected-KV GB/s (fraction of B300 HBM peak) per layer"
# (cache workload, trace workload); "-host": the cache in pinned host memory, recalled per step
WORKLOADS = {"llama3.1-8b-32k": (2, 4), "qwen3-4b-128k": (3, 5), "qwen3-4b-128k-host": (3, 5)}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# ---------------------------------------------------------------- distributed


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: int, seconds_per_rank: float, world: int):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    t = max_over_ranks(seconds_per_rank, world)
    return units_per_rank * world / t, t


def e2e_rates(torch, stream, world, calls, warm, enqueue, out_shape):
    """End to end through a public call with host buffers, two ways, each
    after `warm` untimed steps: (pipelined, synchronised) steps/s.

    enqueue(i, out_host) enqueues step i, which takes its q from pinned host
    memory and leaves its fp32 output in the pinned buffer out_host.
    Synchronised: the host waits for each step before the next.  Pipelined:
    the host enqueues step i, then waits for step i - 1 (an event) and reads
    a value of its output, so one step is in flight while the host prepares
    the next (two pinned output buffers alternate)."""
    outs = [torch.empty(out_shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    views = [o.numpy() for o in outs]
    evs = [torch.cuda.Event() for _ in range(2)]

    def sync_step(i):
        enqueue(i, outs[0])
        stream.synchronize()
        return float(views[0].flat[0])

    def piped(n):
        acc = 0.0
        for i in range(n):
            enqueue(i, outs[i & 1])
            evs[i & 1].record(stream)
            if i > 0:
                evs[(i - 1) & 1].synchronize()
                acc += float(views[(i - 1) & 1].flat[0])
        evs[(n - 1) & 1].synchronize()
        return acc + float(views[(n - 1) & 1].flat[0])

    rates = []
    for mode in ("pipelined", "sync"):
        if mode == "sync":
            for i in range(warm):
                sync_step(i)
        else:
            piped(warm)
        barrier(world)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        if mode == "sync":
            for i in range(calls):
                sync_step(i)
        else:
            piped(calls)
        rates.append(aggregate(calls, time.perf_counter() - w0, world)[0])
    return rates[0], rates[1]


def copy_enqueue(q_host, q_dev, step, out):
    """enqueue() for a step without a host-buffer form: q copied in from
    pinned memory and the output copied back by the copy engines."""
    n_q = q_host.shape[0]

    def enqueue(i, out_host):
        q_dev.copy_(q_host[i % n_q], non_blocking=True)
        step(i, q_dev)
        out_host.copy_(out, non_blocking=True)
    return enqueue


# ---------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.path = None
        self.f = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:                  # no nvidia-smi: the line carries no clock record
            self.proc = None
            if self.f is not None:
                self.f.close()
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 7:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mxs = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mxs) if mxs else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- oracle leg


SEGMENT = 8  # speculative steps per oracle call of the CPU baseline


def cpu_baseline(wl_name: str, seconds: float = 12.0, with_case=False):
    """The fp64 oracle (as it stands) on this host: speculative decode steps
    of the workload's query trace (decision, selection and attention;
    summaries precomputed), in segments of SEGMENT steps (each segment starts
    from an empty state, so its first step corrects every head), until
    `seconds`."""
    import oracle
    from kv_cache_page_build_b300 import synth
    cid, tid = WORKLOADS[wl_name]
    case = synth.make_case(cid)
    wl_trace = synth.WORKLOADS[tid]
    tr = synth.make_trace(wl_trace, case)
    summ = oracle.summaries(case.k_pool, case.page_table)
    wl = case.wl
    cores = oracle.max_threads()
    T = tr.q.shape[0]

    def run(budget):
        n, t0 = 0, time.perf_counter()
        while True:
            i = (n // SEGMENT * SEGMENT) % T
            seg = tr.q[i:i + SEGMENT]
            oracle.speculative_trace(seg, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k,
                                     wl_trace.tau, summ=summ)
            n += seg.shape[0]
            el = time.perf_counter() - t0
            if el >= budget:
                return n, el

    n, el = run(seconds)
    # the same oracle on one thread, for a third of the budget
    oracle.set_threads(1)
    try:
        n1, el1 = run(seconds / 3)
    finally:
        oracle.set_threads(cores)
    res = {"value": n / el, "unit": "steps/s", "cores": cores, "kind": "oracle",
           "sample": f"{n} speculative decode steps (batch {wl.batch}; decision, selection and attention; fp64) "
                     f"of the same workload's query trace in segments of {SEGMENT} steps, in {el:.1f} s; "
                     f"summaries built beforehand",
           "single_thread": {"value": round(n1 / el1, 3), "unit": "steps/s", "cores": 1,
                             "sample": f"{n1} steps in {el1:.1f} s"}}
    return (res, workload_keys(wl_name, wl, wl_trace.tau)) if with_case else res


# ---------------------------------------------------------------- GPU leg


def traffic_for(kernel: str, wl_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel's current source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{wl_name}.traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# What a kernel's DRAM traffic per launch depends on: its device code and
# the host functions that choose its launch shape and tensor maps.
KERNEL_SOURCES = {
    "k_sparse_decode": (("attention.cuh", "common.cuh"),
                        ("make_pool_map", "attn_cluster_size", "launch_attn_gp", "launch_attn_g",
                         "launch_attn")),
}


def _code(text: str) -> str:
    """C/C++ text with comments dropped and whitespace collapsed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def _function(code: str, name: str) -> str:
    """The definition of function `name` in collapsed code: from its return
    type to its closing brace (the first `name(` followed by a body)."""
    import re
    for m in re.finditer(r"\b" + re.escape(name) + r" ?\(", code):
        i = m.end()
        depth = 1
        while i < len(code) and depth:
            depth += {"(": 1, ")": -1}.get(code[i], 0)
            i += 1
        j = i
        while j < len(code) and code[j] not in "{;":
            j += 1
        if j >= len(code) or code[j] != "{":
            continue                               # a call or a declaration
        depth, k = 1, j + 1
        while k < len(code) and depth:
            depth += {"{": 1, "}": -1}.get(code[k], 0)
            k += 1
        start = code.rfind(";", 0, m.start())
        start = max(start, code.rfind("}", 0, m.start())) + 1
        return code[start:k]
    raise KeyError(name)


def kernel_source_hash(kernel: str, read=None) -> str:
    """Hash of what the kernel's traffic depends on (KERNEL_SOURCES), plus
    the status bits of the C header; comments and whitespace are ignored, so
    an edit of the prose alone keeps a profile's counters current.  `read`
    maps a repository path to its text (default: the working tree)."""
    import re
    if read is None:
        def read(rel):
            with open(os.path.join(ROOT, rel)) as f:
                return f.read()
    files, funcs = KERNEL_SOURCES[kernel]
    h = hashlib.sha256()
    for name in files:
        h.update(_code(read(f"kv_cache_page_build_b300/csrc/{name}")).encode())
    host = _code(read("kv_cache_page_build_b300/csrc/kvr.cu"))
    for fn in funcs:
        h.update(_function(host, fn).encode())
    for line in read("include/kvr.h").splitlines():
        if re.match(r"#define KVR_ST_", line):
            h.update(_code(line).encode())
    return h.hexdigest()


def _clock_sampler(dev, local):
    import torch
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    return ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or local))


def _graph_time(torch, g, launches_per_replay, min_launches):
    """Mean device time per launch of a graph of `launches_per_replay` calls,
    replayed back to back (after two untimed replays) until at least
    `min_launches` launches have run; CUDA events around the replays."""
    reps = max(1, -(-min_launches // launches_per_replay))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / (reps * launches_per_replay), reps * launches_per_replay


def measure_hbm(wl_name, args, world, local, steps, warmup, e2e_calls, kernel_launches, clocks=True):
    """One HBM-resident workload: speculative decode steps (selection, then
    attention) over `copies` rotating copies of the cache, timed from a CUDA
    graph; per-kernel times from graphs of back-to-back calls; end-to-end
    eager calls with host copies; the decode-time append.  Returns a dict of
    raw measurements (seconds, bytes)."""
    import torch
    from kv_cache_page_build_b300 import kvr, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cid, tid = WORKLOADS[wl_name]
    COPIES = max(1, args.copies)
    wl_trace = synth.WORKLOADS[tid]
    case = synth.make_case(cid)
    tr = synth.make_trace(wl_trace, case)
    wl = case.wl
    B, Hq, H, D, P, N, k = (wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.n_pages,
                            wl.top_k)
    d = kvr.kvr_dims(**wl.dims())

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    k_pools = [to_dev(case.k_pool.view(np.int16)) for _ in range(COPIES)]
    v_pools = [to_dev(case.v_pool.view(np.int16)) for _ in range(COPIES)]
    page_table = to_dev(case.page_table)
    qs = to_dev(tr.q.view(np.int16))                               # [T][B][Hq][D]
    q_host = torch.from_numpy(tr.q.view(np.int16).copy()).pin_memory()
    TRACE_LEN = qs.shape[0]
    summs = [torch.empty((B, H, N, 2, D), dtype=torch.int16, device=dev) for _ in range(COPIES)]
    del case

    # summaries (prefill-time): one build per copy, timed together
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kvr.kvr_build_summaries(d, k_pools[0], page_table, summs[0])
    torch.cuda.synchronize()
    e0.record()
    for c in range(COPIES):
        kvr.kvr_build_summaries(d, k_pools[c], page_table, summs[c])
    e1.record()
    torch.cuda.synchronize()
    summ_s = e0.elapsed_time(e1) / 1e3 / COPIES

    # speculative state and outputs
    q_prev = torch.zeros((B, Hq, D), dtype=torch.int16, device=dev)
    sel_prev = torch.zeros((B, H, k), dtype=torch.int32, device=dev)
    st = kvr.kvr_spec_state(q_prev.data_ptr(), sel_prev.data_ptr(), 0)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    corrected = torch.empty((B, H), dtype=torch.uint8, device=dev)
    sel_used = torch.empty((B, H, k), dtype=torch.int32, device=dev)
    sel_used_phys = torch.empty((B, H, k), dtype=torch.int32, device=dev)
    ws_n = kvr.kvr_workspace_size(d, k, kvr.KVR_OP_SELECT)
    wa_n = kvr.kvr_workspace_size(d, k, kvr.KVR_OP_ATTN)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=dev)
    wa = torch.zeros(wa_n, dtype=torch.uint8, device=dev)

    def select_call(i):
        kvr.kvr_speculative_select(d, st, qs[i % TRACE_LEN], summs[i % COPIES], page_table, k, wl_trace.tau,
                                   corrected, None, sel_used, sel_used_phys, ws, ws_n)

    def attn_call(i):
        c = i % COPIES
        kvr.kvr_sparse_decode_attn(d, qs[i % TRACE_LEN], k_pools[c], v_pools[c], sel_used_phys, k, 0.0, out,
                                   wa, wa_n)

    side = torch.cuda.Stream()
    ev_d, ev_s = torch.cuda.Event(), torch.cuda.Event()
    ev_d.record()
    ev_s.record()
    wstep = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_STEP), dtype=torch.uint8, device=dev)

    def step(i, q=None):
        c = i % COPIES
        qq = qs[i % TRACE_LEN] if q is None else q
        if args.step == "overlap":
            kvr.kvr_speculative_step_overlap(d, st, qq, summs[c], page_table, k_pools[c], v_pools[c], k,
                                             wl_trace.tau, 0.0, out, corrected, None, sel_used, sel_used_phys,
                                             wstep, wstep.numel(), torch.cuda.current_stream(), side, ev_d,
                                             ev_s)
        else:
            kvr.kvr_speculative_step(d, st, qq, summs[c], page_table, k_pools[c], v_pools[c], k, wl_trace.tau,
                                     0.0, out, corrected, None, sel_used, sel_used_phys, wstep, wstep.numel())

    # warm-up: eager steps (the first one is step 0 of the trace)
    for i in range(max(warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    assert kvr.kvr_get_status() == 0

    # the timed steps: a graph of L steps replayed steps // L times, plus a
    # graph of the remainder, so that exactly `steps` steps run
    L = min(64, steps)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(L):
            step(i)
    rem = steps % L
    graph_rem = None
    if rem:
        graph_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_rem):
            for i in range(rem):
                step(i)
    for _ in range(2):
        graph.replay()
        if graph_rem is not None:
            graph_rem.replay()
    torch.cuda.synchronize()
    reps = steps // L
    sampler = _clock_sampler(dev, local) if clocks else None
    if sampler is not None:
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    # untimed replays enqueued right before the timed ones, so the GPU runs
    # at its working clocks when the timed region starts (no idle gap)
    for _ in range(max(1, -(-256 // L))):
        graph.replay()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        graph.replay()
    if graph_rem is not None:
        graph_rem.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = sampler.stop() if sampler is not None else None
    elapsed = t0.elapsed_time(t1) / 1e3
    status = kvr.kvr_get_status()
    value, t_max = aggregate(steps, elapsed, world)

    # per-launch device time of the selection and of the attention: graphs
    # of 64 back-to-back calls of each kind, replayed until at least
    # `kernel_launches` calls have run
    LK = 64
    graph_sel = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_sel):
        for i in range(LK):
            select_call(i)
    graph_attn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_attn):
        for i in range(LK):
            attn_call(i)
    attn_avg, n_attn = _graph_time(torch, graph_attn, LK, kernel_launches)
    sel_avg, n_sel = _graph_time(torch, graph_sel, LK, kernel_launches)
    status |= kvr.kvr_get_status()

    # several query tokens per step (kvr_sparse_decode_attn_multi): the T
    # newest tokens of every (full) sequence query the same selected pages,
    # so the bytes stay those of one query; T = 1 also with the bf16 store
    seq_full = torch.full((B,), N * P, dtype=torch.int32, device=dev)
    multi = {}
    for T, dt in ((1, kvr.KVR_DTYPE_F32), (1, kvr.KVR_DTYPE_BF16), (2, kvr.KVR_DTYPE_F32), (4, kvr.KVR_DTYPE_F32)):
        qm = qs[:T].permute(1, 0, 2, 3).contiguous()           # [B][T][Hq][D]
        selm = torch.empty((B, H, k), dtype=torch.int32, device=dev)
        selpm = torch.empty_like(selm)
        kvr.kvr_select_pages_multi(d, qm, T, summs[0], page_table, seq_full, k, selm, selpm, None, ws, ws_n)
        out_m = torch.empty((B, T, Hq, D), dtype=torch.float32 if dt == kvr.KVR_DTYPE_F32 else torch.int16,
                            device=dev)
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm):
            for i in range(LK):
                c = i % COPIES
                kvr.kvr_sparse_decode_attn_multi(d, qm, T, k_pools[c], v_pools[c], page_table, seq_full, selm, selpm,
                                                 k, 0.0, out_m, dt, wa, wa_n)
        t_m, _ = _graph_time(torch, gm, LK, kernel_launches)
        multi[f"T={T}" + (" bf16" if dt == kvr.KVR_DTYPE_BF16 else "")] = t_m
    status |= kvr.kvr_get_status()

    # end to end through the public entry point with host buffers: every
    # step takes its q from pinned host memory and leaves its output there
    if args.step == "overlap":  # no host-buffer form: copy-engine transfers
        q_dev = torch.empty((B, Hq, D), dtype=torch.int16, device=dev)
        enqueue = copy_enqueue(q_host[:TRACE_LEN], q_dev, step, out)
    else:
        w_host = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_STEP_HOST), dtype=torch.uint8, device=dev)

        def enqueue(i, out_host):
            c = i % COPIES
            kvr.kvr_speculative_step_host(d, st, q_host[i % TRACE_LEN], summs[c], page_table, k_pools[c],
                                          v_pools[c], k, wl_trace.tau, 0.0, out_host, corrected, None, sel_used,
                                          sel_used_phys, w_host, w_host.numel())
    e2e_value, e2e_sync = e2e_rates(torch, torch.cuda.current_stream(), world, e2e_calls, 200, enqueue,
                                    (B, Hq, D))
    status |= kvr.kvr_get_status()

    # decode-time append (kvr_append_kv), timed last: a graph of LK appends
    # into the last LK token slots of cache copy 0 (its lengths set LK tokens
    # short), re-armed and replayed
    app_len = torch.full((B,), N * P - LK, dtype=torch.int32, device=dev)
    k_rows = torch.zeros((B, H, D), dtype=torch.int16, device=dev)
    graph_app = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_app):
        for _ in range(LK):
            kvr.kvr_append_kv(d, k_rows, k_rows, page_table, app_len, k_pools[0], v_pools[0], summs[0])
    app_times = []
    for _ in range(6):
        app_len.fill_(N * P - LK)
        torch.cuda.synchronize()
        ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ta.record()
        graph_app.replay()
        tb.record()
        torch.cuda.synchronize()
        app_times.append(ta.elapsed_time(tb) / 1e3 / LK)
    app_avg = statistics.median(app_times[1:])
    status |= kvr.kvr_get_status()
    res = dict(wl=wl, tau=wl_trace.tau, copies=COPIES, steps=steps, L=L, value=value, t_max=t_max,
               attn_avg=attn_avg, n_attn=n_attn, sel_avg=sel_avg, n_sel=n_sel, app_avg=app_avg, summ_s=summ_s,
               multi=multi,
               e2e_value=e2e_value, e2e_sync=e2e_sync, e2e_calls=e2e_calls, clk=clk, status=status,
               attn_bytes=B * H * k * P * 2 * D * 2,          # selected K and V rows read per launch
               summ_bytes=B * H * N * 2 * D * 2,               # summaries read by the selection
               k_bytes=B * N * P * H * D * 2)
    del k_pools, v_pools, summs, qs
    torch.cuda.empty_cache()
    return res


def hbm_kernels(r):
    """The per-kernel figures of one HBM workload."""
    hbm, _ = peaks()
    gbs = r["attn_bytes"] / r["attn_avg"] / 1e9
    sel_gbs = r["summ_bytes"] / r["sel_avg"] / 1e9
    wl = r["wl"]
    build_bytes = r["k_bytes"] + r["summ_bytes"]
    return {
        "attention (k_sparse_decode)": {"us": round(r["attn_avg"] * 1e6, 3), "bytes": r["attn_bytes"],
                                        "gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                                        "launches_timed": r["n_attn"]},
        "selection (k_page_scores + k_topk)": {"us": round(r["sel_avg"] * 1e6, 3), "bytes": r["summ_bytes"],
                                               "gbs": round(sel_gbs, 1), "frac": round(sel_gbs / hbm, 4),
                                               "launches_timed": r["n_sel"]},
        "k_append (decode-time append, one token per sequence)": {
            "us": round(r["app_avg"] * 1e6, 3), "bytes": wl.batch * wl.n_kv_heads * (2 * wl.head_dim * 2 +
                                                                                    2 * 2 * wl.head_dim * 2),
            "note": "latency-bound: K and V rows written and the page summary read and written per "
                    "(sequence, KV head)"},
        "k_build_summaries": {"us": round(r["summ_s"] * 1e6, 3), "bytes": build_bytes,
                              "gbs": round(build_bytes / r["summ_s"] / 1e9, 1),
                              "note": "once per cache (prefill), not in the step"},
        "several queries per step (k_sparse_decode, kvr_sparse_decode_attn_multi)": {
            name: {"us": round(t * 1e6, 3), "gbs": round(r["attn_bytes"] / t / 1e9, 1),
                   "frac": round(r["attn_bytes"] / t / 1e9 / hbm, 4),
                   "vs_one_query": round(t / r["multi"]["T=1"], 3)}
            for name, t in r["multi"].items()},
    }


def workload_keys(name, wl, tau):
    """The config keys that name a workload (shared by both arms' lines)."""
    B, Hq, H, D, P, k = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.top_k
    return {
        "workload": f"{name}: {B} sequences x {Hq}/{H} heads, head_dim {D}, context {wl.context}, page {P}, "
                    f"top-k {k} pages; speculative, tau {tau}",
        "batch": B, "n_q_heads": Hq, "n_kv_heads": H, "head_dim": D, "context": wl.context, "page_size": P,
        "top_k": k, "tau": tau, "storage": "bf16",
    }


def hbm_config(name, r, world):
    return {
        **workload_keys(name, r["wl"], r["tau"]),
        "accumulate": "f32",
        "parallelism": f"{world} independent replica(s)" if world > 1 else "1 GPU",
        "l2": f"{r['copies']} rotating cache copies: "
              f"{(r['copies'] - 1) * (r['attn_bytes'] + r['summ_bytes']) / 2**20:.0f} MiB touched between reuses "
              f"of one copy (L2 126 MB)",
        "graph": f"steps replayed from a CUDA graph of {r['L']} steps; per-kernel times from graphs of 64 "
                 f"back-to-back calls of each kind, {r['n_attn']} attention and {r['n_sel']} selection launches "
                 f"timed",
    }


def hbm_summary(name, r):
    """A compact record of a workload that is not the line's headline."""
    hbm, _ = peaks()
    gbs = r["attn_bytes"] / r["attn_avg"] / 1e9
    return {"workload": hbm_config(name, r, 1)["workload"], "steps_per_s": round(r["value"], 2),
            "steps": r["steps"], "ms_per_step": round(r["t_max"] / r["steps"] * 1e3, 5),
            "roofline": {"bound": "hbm", "kernel": "k_sparse_decode", "achieved": round(gbs, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(gbs / hbm, 4)},
            "kernels": hbm_kernels(r),
            "e2e_steps_per_s": round(r["e2e_value"], 2), "clocks": r["clk"], "device_status": r["status"]}


def measure_recall(args, world, local, reps, warmup, e2e_calls, clocks=True):
    """The host-resident workload: the K/V cache in page-locked host memory
    (head-major), summaries and a 2k-slot working set per (sequence, KV head)
    in HBM; each step selects speculatively, recalls the missing pages on a
    side stream and attends over the working set (kvr_speculative_step_recall).
    Steps replay from a CUDA graph of the 32-step query trace, `reps` times."""
    import torch
    from kv_cache_page_build_b300 import kvr, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cid, tid = WORKLOADS["qwen3-4b-128k-host"]
    wl_trace = synth.WORKLOADS[tid]
    case = synth.make_case(cid)
    tr = synth.make_trace(wl_trace, case)
    wl = case.wl
    B, Hq, H, D, P, N, k = (wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.n_pages,
                            wl.top_k)
    S = 2 * k
    d = kvr.kvr_dims(**wl.dims())
    page_bytes = 2 * P * D * 2                      # K and V of one (sequence, head, page)

    # prefill: the summaries come from a device copy of K; the head-major
    # host copy of K and V is laid out on the device and copied to
    # page-locked host memory, then the device copies are dropped
    page_table = torch.from_numpy(case.page_table).to(dev)
    summ = torch.empty((B, H, N, 2, D), dtype=torch.int16, device=dev)
    host_pools = []
    for pool in (case.k_pool, case.v_pool):
        p_dev = torch.from_numpy(pool.view(np.int16)).to(dev)
        if not host_pools:
            kvr.kvr_build_summaries(d, p_dev, page_table, summ)
        hnd = p_dev[page_table.reshape(-1).long()].view(B, N, P, H, D).permute(0, 3, 1, 2, 4).contiguous()
        h = torch.empty(hnd.shape, dtype=torch.int16).pin_memory()
        h.copy_(hnd)
        host_pools.append(h)
        del p_dev, hnd
    torch.cuda.synchronize()
    k_host, v_host = host_pools
    del case
    torch.cuda.empty_cache()
    k_slots = torch.zeros((B, S, P, H, D), dtype=torch.int16, device=dev)
    v_slots = torch.zeros_like(k_slots)
    p2s = torch.empty((B, H, N), dtype=torch.int32, device=dev)
    s2p = torch.empty((B, H, S), dtype=torch.int32, device=dev)
    host = kvr.kvr_host_kv(k_host.data_ptr(), v_host.data_ptr())
    wset = kvr.kvr_working_set(k_slots.data_ptr(), v_slots.data_ptr(), p2s.data_ptr(), s2p.data_ptr(), S)
    qs = torch.from_numpy(tr.q.view(np.int16).copy()).to(dev)   # [T][B][Hq][D]
    q_host = torch.from_numpy(tr.q.view(np.int16).copy()).pin_memory()
    T = qs.shape[0]
    main_s = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ev_s, ev_r = torch.cuda.Event(), torch.cuda.Event()
    ev_s.record()
    ev_r.record()

    def timed(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = None
        for _ in range(n):
            torch.cuda.synchronize()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b) / 1e3
            best = t if best is None else min(best, t)
        return best

    # the host link: one pinned 1 GiB host-to-device copy (best of 3)
    link_dst = torch.empty(k_host.numel(), dtype=torch.int16, device=dev)
    link_s = timed(lambda: link_dst.copy_(k_host.view(-1), non_blocking=True), 3)
    link_gbs = k_host.numel() * 2 / link_s / 1e9
    del link_dst

    # the recall kernel on a cold working set: every page of a full selection is missing
    sel0 = torch.empty((B, H, k), dtype=torch.int32, device=dev)
    wsel = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_SELECT), dtype=torch.uint8, device=dev)
    kvr.kvr_select_pages(d, qs[0], summ, page_table, k, sel0, None, None, wsel, wsel.numel())
    n_copied = torch.zeros(1, dtype=torch.int32, device=dev)
    recall_times = []
    for _ in range(5):
        kvr.kvr_working_set_reset(d, wset)
        torch.cuda.synchronize()
        recall_times.append(timed(lambda: kvr.kvr_recall_pages(d, host, wset, sel0, sel0, None, k, None,
                                                                n_copied), 1))
    recall_s = min(recall_times)
    recall_bytes = B * H * k * page_bytes

    # speculative steps with recall, replayed from a CUDA graph of T steps
    q_prev = torch.zeros((B, Hq, D), dtype=torch.int16, device=dev)
    sel_prev = torch.zeros((B, H, k), dtype=torch.int32, device=dev)
    st = kvr.kvr_spec_state(q_prev.data_ptr(), sel_prev.data_ptr(), 0)
    out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    corrected = torch.empty((B, H), dtype=torch.uint8, device=dev)
    sel_used = torch.empty((B, H, k), dtype=torch.int32, device=dev)
    sel_used_slot = torch.empty((B, H, k), dtype=torch.int32, device=dev)
    ws = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_STEP), dtype=torch.uint8, device=dev)

    def step(i, q=None):
        kvr.kvr_speculative_step_recall(d, st, qs[i % T] if q is None else q, summ, host, wset, k,
                                        wl_trace.tau, 0.0, out, corrected, None, sel_used, sel_used_slot,
                                        n_copied, ws, ws.numel(), torch.cuda.current_stream(), side, ev_s,
                                        ev_r)

    kvr.kvr_working_set_reset(d, wset)
    for i in range(max(warmup, 3)):     # step 0 of the trace first (every head corrected)
        step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        for i in range(T):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    sampler = _clock_sampler(dev, local) if clocks else None
    if sampler is not None:
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    graph.replay()                      # untimed, right before the timed replays
    torch.cuda.synchronize()
    n0 = int(n_copied.item())
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = sampler.stop() if sampler is not None else None
    elapsed = t0.elapsed_time(t1) / 1e3
    n_steps = reps * T
    pages_per_step = (int(n_copied.item()) - n0) / n_steps
    value, t_max = aggregate(n_steps, elapsed, world)
    status = kvr.kvr_get_status()

    # end to end through the public call: q in from pinned memory, output
    # back, every step
    q_dev = torch.empty((B, Hq, D), dtype=torch.int16, device=dev)
    e2e_value, e2e_sync = e2e_rates(torch, main_s, world, e2e_calls, 16, copy_enqueue(q_host[:T], q_dev, step, out),
                                    (B, Hq, D))
    status |= kvr.kvr_get_status()
    res = dict(wl=wl, tau=wl_trace.tau, S=S, T=T, steps=n_steps, value=value, t_max=t_max,
               pages_per_step=pages_per_step, page_bytes=page_bytes, recall_s=recall_s,
               recall_bytes=recall_bytes, link_gbs=link_gbs, e2e_value=e2e_value, e2e_sync=e2e_sync,
               e2e_calls=e2e_calls,
               clk=clk, status=status)
    del k_slots, v_slots, k_host, v_host, host_pools
    torch.cuda.empty_cache()
    return res


def recall_roofline(r):
    gbs = r["recall_bytes"] / r["recall_s"] / 1e9
    return {"bound": "host_link", "achieved": round(gbs, 1), "peak": round(r["link_gbs"], 1), "unit": "GB/s",
            "frac": round(gbs / r["link_gbs"], 4), "traffic": None,
            "peak_kind": "measured in this run: pinned 1 GiB host-to-device copy, best of 3",
            "kernel": "k_recall", "bytes_per_launch": r["recall_bytes"],
            "launch_us": round(r["recall_s"] * 1e6, 3),
            "how": "cold working set: all B*H*k pages of one selection recalled in one launch"}


def recall_workload(r):
    wl = r["wl"]
    return (f"qwen3-4b-128k-host: {wl.batch} sequences x {wl.n_q_heads}/{wl.n_kv_heads} heads, head_dim "
            f"{wl.head_dim}, context {wl.context}, page {wl.page_size}, top-k {wl.top_k} pages; K/V in "
            f"page-locked host memory (head-major), {r['S']}-slot working set per (sequence, KV head) in HBM; "
            f"speculative, tau {r['tau']}")


def recall_summary(r):
    return {"workload": recall_workload(r), "steps_per_s": round(r["value"], 2), "steps": r["steps"],
            "ms_per_step": round(r["t_max"] / r["steps"] * 1e3, 5),
            "recalled_pages_per_step": round(r["pages_per_step"], 2),
            "recalled_gbs_per_step_rate": round(r["pages_per_step"] * r["page_bytes"] * r["value"] / 1e9, 2),
            "roofline": recall_roofline(r), "e2e_steps_per_s": round(r["e2e_value"], 2),
            "clocks": r["clk"], "device_status": r["status"]}


def hbm_line(name, r, args, world):
    """The JSON line of an HBM-resident workload as the headline."""
    hbm, peak_kind = peaks()
    achieved = r["attn_bytes"] / r["attn_avg"] / 1e9
    wl = r["wl"]
    B, Hq, D = wl.batch, wl.n_q_heads, wl.head_dim
    cfg = hbm_config(name, r, world)
    cfg["step"] = f"kvr_speculative_step{'_overlap' if args.step == 'overlap' else ''}"
    return {
        "metric": METRIC,
        "value": round(r["value"], 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": r["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(r["t_max"] / r["steps"] * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": cfg,
        "selected_kv_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic_for("k_sparse_decode", name),
                     "peak_kind": peak_kind, "kernel": "k_sparse_decode", "bytes_per_launch": r["attn_bytes"],
                     "launch_us": round(r["attn_avg"] * 1e6, 3), "launches_timed": r["n_attn"]},
        "kernels": hbm_kernels(r),
        # k_page_scores, k_topk, k_sparse_decode (+ k_spec_decide and a second attention launch)
        "gpu_launches": (5 if args.step == "overlap" else 3) * r["steps"],
        "e2e": {"value": round(r["e2e_value"], 2), "unit": "steps/s",
                "h2d_bytes_per_step": B * Hq * D * 2, "d2h_bytes_per_step": B * Hq * D * 4,
                "synchronised_per_step": round(r["e2e_sync"], 2),
                "how": (f"{r['e2e_calls']} eager kvr_speculative_step_overlap calls after 200 untimed ones, q "
                        f"copied in from pinned host memory and the fp32 output copied back by the copy engines "
                        f"every step"
                        if args.step == "overlap" else
                        f"{r['e2e_calls']} eager kvr_speculative_step_host calls after 200 untimed ones: every "
                        f"step reads its q from pinned host memory (staged by its first kernel) and the "
                        f"attention writes the fp32 output into pinned host memory")
                       + "; pipelined: the host enqueues step i, then waits for step i-1 and reads its output "
                         "(one step in flight); synchronised_per_step: the host waits for each step"},
        "clocks": r["clk"],
        "device_status": r["status"],
    }


def recall_line(r, args, world):
    """The JSON line of the host-resident workload as the headline."""
    wl = r["wl"]
    B, Hq, D = wl.batch, wl.n_q_heads, wl.head_dim
    return {
        "metric": METRIC,
        "value": round(r["value"], 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": r["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(r["t_max"] / r["steps"] * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": recall_workload(r),
            "batch": B, "n_q_heads": Hq, "n_kv_heads": wl.n_kv_heads, "head_dim": D, "context": wl.context,
            "page_size": wl.page_size, "top_k": wl.top_k, "tau": r["tau"], "storage": "bf16",
            "accumulate": "f32",
            "parallelism": f"{world} independent replica(s)" if world > 1 else "1 GPU",
            "l2": "the host cache (2 GiB) does not fit L2; each recalled page is read from host memory once",
            "graph": f"steps replayed from a CUDA graph of {r['T']} steps (the {r['T']}-step query trace, "
                     f"repeated)",
        },
        "recalled_pages_per_step": round(r["pages_per_step"], 2),
        "roofline": recall_roofline(r),
        "gpu_launches": 5 * r["steps"],  # k_page_scores, k_topk, k_recall, k_sparse_decode x2
        "e2e": {"value": round(r["e2e_value"], 2), "unit": "steps/s",
                "h2d_bytes_per_step": B * Hq * D * 2, "d2h_bytes_per_step": B * Hq * D * 4,
                "synchronised_per_step": round(r["e2e_sync"], 2),
                "how": f"{r['e2e_calls']} eager kvr_speculative_step_recall calls after 16 untimed ones, q "
                       f"copied in from pinned host memory and the fp32 output copied back every step; "
                       f"pipelined: one step in flight while the host reads the previous step's output; "
                       f"synchronised_per_step: the host waits for each step"},
        "clocks": r["clk"],
        "device_status": r["status"],
    }


def run_gpu(args, world, rank, local):
    """The line of --workload, plus (unless --no-extras) compact records of
    the other HBM-resident workload and of the host-resident one."""
    e2e_calls = max(1, args.e2e_calls)
    if args.workload.endswith("-host"):
        r = measure_recall(args, world, local, reps=max(1, -(-args.steps // 32)), warmup=args.warmup,
                           e2e_calls=e2e_calls)
        return recall_line(r, args, world)
    r = measure_hbm(args.workload, args, world, local, args.steps, args.warmup, e2e_calls,
                    kernel_launches=args.kernel_launches)
    line = hbm_line(args.workload, r, args, world)
    if not args.no_extras:
        other = "llama3.1-8b-32k" if args.workload == "qwen3-4b-128k" else "qwen3-4b-128k"
        r2 = measure_hbm(other, args, world, local, 640, args.warmup, 1000,
                         kernel_launches=args.kernel_launches, clocks=True)
        line["also"] = {other: hbm_summary(other, r2)}
        rr = measure_recall(args, world, local, reps=8, warmup=args.warmup, e2e_calls=96)
        line["also"]["qwen3-4b-128k-host"] = recall_summary(rr)
    return line


# ---------------------------------------------------------------- multi-layer pipeline

# bf16 weight bytes one decode step reads per transformer layer: (QKV
# projection, output projection + gated FFN); the pipeline's stand-in reads
# as many.  Llama-3.1-8B: hidden 4096, 32/8 heads of 128, FFN 14336.
# Qwen3-4B: hidden 2560, 32/8 heads of 128, FFN 9728.
MODEL_BYTES = {
    "llama3.1-8b-32k": (4096 * (4096 + 2 * 1024) * 2, (4096 * 4096 + 3 * 4096 * 14336) * 2),
    "qwen3-4b-128k": (2560 * (4096 + 2 * 1024) * 2, (4096 * 2560 + 3 * 2560 * 9728) * 2),
}
MODEL_BYTES["qwen3-4b-128k-host"] = MODEL_BYTES["qwen3-4b-128k"]

BREAKDOWN = (("qkv_stand_in", 0, 1), ("selection_main", 1, 2), ("attention_reused", 2, 3),
             ("exposed_wait", 3, 4), ("attention_corrected", 4, 5), ("post_stand_in", 5, 6),
             ("layer_total", 0, 6), ("side_stream", 7, 8), ("prefetch_stream", 9, 10))


def run_gpu_pipeline(args, world, rank, local):
    """A decode step through --layers attention layers with kvr_pipeline_step.
    Each layer has its own copy of the workload's cache (in HBM, or in
    page-locked host memory for the -host workload), its own summaries,
    state and working set, and its own phase of the query trace; the
    stand-in reads the model's projection weights (one buffer shared by the
    layers, larger than L2) before and after each attention.  Timed from a
    CUDA graph of steps; the latency breakdown comes from an eager run with
    the pipeline's timing marks; the same layers stepped one at a time
    (kvr_speculative_step, or kvr_speculative_step_recall, between the same
    stand-in reads) are timed beside it."""
    import types
    import torch
    from kv_cache_page_build_b300 import kvr, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cid, tid = WORKLOADS[args.workload]
    host_mode = args.workload.endswith("-host")
    wl_trace = synth.WORKLOADS[tid]
    case = synth.make_case(cid)
    tr = synth.make_trace(wl_trace, case)
    wl = case.wl
    B, Hq, H, D, P, N, k = (wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.n_pages,
                            wl.top_k)
    S, nL, tau = 2 * k, args.layers, wl_trace.tau
    d = kvr.kvr_dims(**wl.dims())
    qs = torch.from_numpy(tr.q.view(np.int16).copy()).to(dev)
    T = qs.shape[0]
    page_table = torch.from_numpy(case.page_table).to(dev)
    k0 = torch.from_numpy(case.k_pool.view(np.int16)).to(dev)
    summ0 = torch.empty((B, H, N, 2, D), dtype=torch.int16, device=dev)
    kvr.kvr_build_summaries(d, k0, page_table, summ0)
    torch.cuda.synchronize()
    if host_mode:
        del k0
        kh, vh = synth.host_hnd(case)
        caches = [(torch.from_numpy(kh.view(np.int16)).pin_memory(), torch.from_numpy(vh.view(np.int16)).pin_memory())
                  for _ in range(nL)]
        del kh, vh
    else:
        v0 = torch.from_numpy(case.v_pool.view(np.int16)).to(dev)
        caches = [(k0.clone(), v0.clone()) for _ in range(nL)]
        del k0, v0
    del case
    summs = [summ0.clone() for _ in range(nL)]
    del summ0
    qkv_b, post_b = MODEL_BYTES[args.workload]
    weights = torch.randint(-2 ** 31, 2 ** 31 - 1, ((qkv_b + post_b) // 4,), dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    compute = kvr.stand_in(weights, qkv_b, post_b, sink)
    # one workspace for the pipeline's layers (it orders their uses) and one for the sequential run
    ws = torch.zeros(kvr.kvr_workspace_size(d, k, kvr.KVR_OP_STEP), dtype=torch.uint8, device=dev)
    ws_seq = torch.zeros_like(ws)

    def events(n, timing=False):
        evs = [torch.cuda.Event(enable_timing=timing) for _ in range(n)]
        for e in evs:
            e.record()
        return evs

    def make_layer(i):
        o = types.SimpleNamespace(summ=summs[i])
        o.q_prev = torch.zeros((B, Hq, D), dtype=torch.int16, device=dev)
        o.sel_prev = torch.zeros((B, H, k), dtype=torch.int32, device=dev)
        o.st = kvr.kvr_spec_state(o.q_prev.data_ptr(), o.sel_prev.data_ptr(), 0)
        o.out = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
        o.corrected = torch.empty((B, H), dtype=torch.uint8, device=dev)
        o.sel_used = torch.empty((B, H, k), dtype=torch.int32, device=dev)
        o.idx = torch.empty((B, H, k), dtype=torch.int32, device=dev)
        o.ev = events(3)
        o.phase = (7 * i) % T
        if host_mode:
            o.host = kvr.kvr_host_kv(caches[i][0].data_ptr(), caches[i][1].data_ptr())
            o.k_slots = torch.zeros((B, S, P, H, D), dtype=torch.int16, device=dev)
            o.v_slots = torch.zeros_like(o.k_slots)
            o.p2s = torch.empty((B, H, N), dtype=torch.int32, device=dev)
            o.s2p = torch.empty((B, H, S), dtype=torch.int32, device=dev)
            o.wset = kvr.kvr_working_set(o.k_slots.data_ptr(), o.v_slots.data_ptr(), o.p2s.data_ptr(),
                                         o.s2p.data_ptr(), S)
            kvr.kvr_working_set_reset(d, o.wset)
            o.n_copied = torch.zeros(1, dtype=torch.int32, device=dev)
            o.extra = dict(host=o.host, wset=o.wset, n_copied_opt=o.n_copied)
        else:
            o.extra = dict(page_table=page_table, k_pool=caches[i][0], v_pool=caches[i][1])
        return o

    pipe, seq = [make_layer(i) for i in range(nL)], [make_layer(i) for i in range(nL)]
    side, pf = torch.cuda.Stream(), torch.cuda.Stream()

    def pipe_step(i, marks=None):
        io = [kvr.layer(o.st, qs[(i + o.phase) % T], o.summ, o.out, o.corrected, None, o.sel_used, o.idx, ws,
                        ws.numel(), o.ev, **o.extra) for o in pipe]
        kvr.kvr_pipeline_step(d, io, compute, k, tau, 0.0, torch.cuda.current_stream(), side, pf, marks)

    def seq_step(i):
        cur = torch.cuda.current_stream()
        for o in seq:
            q = qs[(i + o.phase) % T]
            kvr.kvr_stand_in_read(compute, 0, qkv_b)
            if host_mode:
                kvr.kvr_speculative_step_recall(d, o.st, q, o.summ, o.host, o.wset, k, tau, 0.0, o.out, o.corrected,
                                                None, o.sel_used, o.idx, o.n_copied, ws_seq, ws_seq.numel(), cur,
                                                side, o.ev[0], o.ev[1])
            else:
                kvr.kvr_speculative_step(d, o.st, q, o.summ, page_table, o.extra["k_pool"], o.extra["v_pool"], k,
                                         tau, 0.0, o.out, o.corrected, None, o.sel_used, o.idx, ws_seq,
                                         ws_seq.numel())
            kvr.kvr_stand_in_read(compute, qkv_b, post_b)

    def join():
        for o in pipe:
            torch.cuda.current_stream().wait_event(o.ev[2])

    for i in range(max(args.warmup, 3)):           # step 0 of each layer's trace phase first
        pipe_step(i)
        seq_step(i)
    torch.cuda.synchronize()
    G = 8

    def capture(fn, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for o in pipe:
                o.ev[2].record()                    # the cross-step wait needs a record inside the capture
            for i in range(first, first + G):
                fn(i)
            join()
        return g

    w0 = max(args.warmup, 3)
    g_pipe, g_seq = capture(pipe_step, w0), capture(seq_step, w0)
    g_pipe.replay()
    g_seq.replay()
    for o in pipe:
        o.ev[2].record()                            # last recorded inside a capture: record it for eager steps
    torch.cuda.synchronize()
    reps = max(1, args.steps // G)

    def timed(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    clocks = _clock_sampler(dev, local)
    time.sleep(0.3)
    barrier(world)
    t_pipe = timed(g_pipe)
    t_seq = timed(g_seq)
    barrier(world)
    clk = clocks.stop()
    n_steps = reps * G
    value, t_max = aggregate(n_steps, t_pipe, world)
    seq_value, t_seq_max = aggregate(n_steps, t_seq, world)

    # latency breakdown: a graph of the same steps that also records the
    # pipeline's timing marks; each replay leaves the times of its last step
    marks = events(nL * kvr.KVR_PIPE_MARKS, timing=True)
    g_mark = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_mark, capture_error_mode="thread_local"):
        for o in pipe:
            o.ev[2].record()
        for i in range(w0, w0 + G):
            pipe_step(i, marks)
        join()
    for o in pipe:
        o.ev[2].record()
    sums = {name: 0.0 for name, _, _ in BREAKDOWN}
    M = 24
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_mark = 0.0
    for _ in range(M):
        torch.cuda.synchronize()
        a_ev.record()
        g_mark.replay()
        b_ev.record()
        torch.cuda.synchronize()
        t_mark += a_ev.elapsed_time(b_ev) / 1e3
        for l in range(nL):
            m = marks[l * kvr.KVR_PIPE_MARKS:(l + 1) * kvr.KVR_PIPE_MARKS]
            for name, a, b in BREAKDOWN:
                sums[name] += m[a].elapsed_time(m[b]) * 1e3
    breakdown = {name: round(v / (M * nL), 2) for name, v in sums.items()}
    status = kvr.kvr_get_status()
    # two stand-ins; host: 2 selection kernels, 2 recalls, 2 attentions; HBM: scores, top-k, attention
    per_layer = 2 + (6 if host_mode else 3)
    return {
        "metric": METRIC + "; here whole multi-layer steps",
        "value": round(value, 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": n_steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / n_steps * 1e3, 5),
        "us_per_layer": round(t_max / n_steps / nL * 1e6, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}, {nL}-layer pipeline: {B} sequences x {Hq}/{H} heads, head_dim {D}, "
                        f"context {wl.context}, page {P}, top-k {k}; cache "
                        + ("in page-locked host memory, recalled into a 2k-slot working set" if host_mode
                           else "in HBM") + f"; speculative, tau {tau}; stand-in reads of {qkv_b} + {post_b} "
                        f"bytes of projection weights per layer",
            "layers": nL, "batch": B, "n_q_heads": Hq, "n_kv_heads": H, "head_dim": D, "context": wl.context,
            "page_size": P, "top_k": k, "tau": tau, "stand_in_bytes": [qkv_b, post_b],
            "parallelism": f"{world} independent replica(s)" if world > 1 else "1 GPU",
            "l2": "each layer's cache is its own copy and the stand-in streams more than L2 between layers",
            "graph": f"steps replayed from a CUDA graph of {G} steps",
        },
        "sequential": {"value": round(seq_value, 2), "unit": "steps/s",
                       "ms_per_step": round(t_seq_max / n_steps * 1e3, 5),
                       "how": "the same layers one call at a time: " + (
                           "kvr_speculative_step_recall" if host_mode else "kvr_speculative_step") +
                       " between the same stand-in reads, from a CUDA graph"},
        "breakdown_us_per_layer": breakdown,
        "step_us_with_marks": round(t_mark / (M * G) * 1e6, 2),
        "breakdown_how": f"a CUDA graph of {G} steps that records the pipeline's timing marks, replayed {M} times; "
                         f"the last step of each replay, mean over {M} x {nL} layers (step_us_with_marks: the "
                         "whole multi-layer step with the marks recorded); HBM layers run their selection and "
                         "attention as one chain of dependent launches (selection_main spans both, the other "
                         "attention spans and both side spans are 0); host layers: side_stream = the corrected "
                         "heads' recall, prefetch_stream = the recall of the other heads' pages for the next step",
        "roofline": None,
        "gpu_launches": per_layer * nL * n_steps,
        "clocks": clk,
        "device_status": status,
    }


# ---------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64000)
    ap.add_argument("--warmup", type=int, default=128)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3-4b-128k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-extras", action="store_true",
                    help="only the --workload line (no records of the other workloads under 'also')")
    ap.add_argument("--kernel-launches", type=int, default=1280,
                    help="launches timed for each per-kernel figure (selection, attention)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-calls", type=int, default=2000,
                    help="timed eager calls of each e2e measurement (after 200 untimed ones)")
    ap.add_argument("--copies", type=int, default=4, help="rotating cache copies (L2-cold timing needs >= 3)")
    ap.add_argument("--step", default="sequential", choices=["sequential", "overlap", "pipeline"],
                    help="kvr_speculative_step, kvr_speculative_step_overlap (selection on a side stream), or "
                         "kvr_pipeline_step over --layers layers with stand-in projections")
    ap.add_argument("--layers", type=int, default=4, help="attention layers of --step pipeline")
    args = ap.parse_args()
    world, rank, local = dist_setup()

    if args.impl == "reference":
        if rank != 0:
            return
        # each timed step is one full oracle decode step; the run is bounded in time
        secs = min(60.0, max(5.0, 0.5 * (args.steps + args.warmup)))
        base, wkeys = cpu_baseline(args.workload, seconds=secs, with_case=True)
        line = {"impl": "reference", "metric": METRIC, "value": round(base["value"], 4), "unit": "steps/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 / base["value"], 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {**wkeys, "accumulate": "f64", "parallelism": "host cores (OpenMP)"},
                "cpu_baseline": base,
                "e2e": {"value": round(base["value"], 4), "unit": "steps/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.step == "pipeline":
        res = run_gpu_pipeline(args, world, rank, local)
    else:
        res = run_gpu(args, world, rank, local)
    if rank == 0:
        if args.step == "pipeline":
            res["cpu_baseline"] = None
        elif world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload)
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res))


if __name__ == "__main__":
    main()
