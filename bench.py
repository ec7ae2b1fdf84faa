"""Benchmark of the sparse-decode hot path on GB300.

Headline: the Quest decode workload with 16 sequences of 32K context (32 query
/ 4 KV heads, head_dim 128, bf16 paged KV, 2048-token budget per KV head).
One step = one decode step of the whole batch: append the new token
(page-summary update), Quest selection (scores + top-k + AttentionView),
split-K decode + LSE merge.  Metric: decode queries/s (one query = one
sequence's step over all query heads), with the decode kernel's achieved HBM
bandwidth against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

L2 is flushed (a 512 MiB write) before every timed step; steps are timed
with CUDA events on the launching stream.  Under torchrun each rank runs an
independent replica (no collective on the data path); rank 0 prints one JSON
line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode-attn queries/s at 1 GB300; achieved HBM GB/s vs peak"
HEADLINE = "quest_32k"
FLUSH_BYTES = 512 << 20
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "kv_cache_decode_quest_gb300", "csrc")
# the Quest step as the bench runs it: "step" = append, select and decode in one
# kernel (se_quest_step); "fused" = se_quest_select_append + se_sparse_decode
HEADLINE_MODE = "step"
RAGGED_MODE = "step"
# the one-query latency line: the two calls are ~2 us faster there (a
# cooperative launch of the whole grid for one unit costs more than it saves)
TINY_MODE = "fused"
# per mode: the dominant kernel, its source and its committed ncu traffic record
KERNEL_OF_MODE = {
    "step": ("quest_step_kernel", os.path.join(CSRC, "quest_step.cu"), "quest_step_kernel_{}.json"),
    "fused": ("decode_kernel", os.path.join(CSRC, "decode.cu"), "decode_kernel_{}.json"),
}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """(dense bf16 TFLOP/s of a GEMM timed alone, SM clock MHz, kind)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("sm_max_mhz", 2070.0)), "measured"
    return 1900.0, 2070.0, "fallback"


# Exponentials per clock per SM: the special-function rate of this GPU
# generation (twice the previous one's 16); with the SM count and the
# maximum SM clock it gives the ex2 roof of the SnapKV scoring passes.
EX2_PER_CLOCK_PER_SM = 32


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(name, src):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, or None
    when the summary is missing or the kernel source changed since."""
    path = os.path.join(PROFILE_DIR, name)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha") != file_sha(src):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# CPU oracle baseline (spawned workers; the oracle as it stands)
# ---------------------------------------------------------------------------

def _oracle_worker(args):
    """Run oracle Quest queries of one sequence for about `seconds`."""
    name, b, seconds = args
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, ROOT)
    import oracle
    from kv_cache_decode_quest_gb300 import synth
    w = synth.workloads()[name]
    k, v = synth.quest_sequence(w, b)
    q = synth.quest_queries(w)
    G = w.num_q_heads // w.num_kv_heads
    scale = 1.0 / math.sqrt(w.head_dim)
    done, t0 = 0, time.perf_counter()
    s = 0
    while True:
        L = w.ctx[b] + s + 1
        for h in range(w.num_kv_heads):
            K = oracle.widen(k[h, :L])
            V = oracle.widen(v[h, :L])
            qg = oracle.widen(q[s, b, h * G:(h + 1) * G])
            U = oracle.quest_bound(qg, *oracle.page_minmax(K))
            pages = oracle.quest_select(U, oracle.quest_k_pages(min(w.budget[b], 2 ** 31 - 1)))
            tok = oracle.quest.selected_tokens(pages, L)
            oracle.attend(qg, K[tok], V[tok], scale)
        done += 1
        s = (s + 1) % w.steps
        if time.perf_counter() - t0 >= seconds:
            break
    return done, time.perf_counter() - t0


def cpu_model():
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu), or the machine type."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def _timed_calls(fn, seconds):
    """Calls fn() until `seconds` have passed (at least once); returns calls/s."""
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return n / dt, n


def _oracle_rates_worker(seconds):
    """Single-threaded oracle rates of one query of each workload (the oracle as
    it stands; a bounded sample of each workload's queries)."""
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    from oracle.quest import selected_tokens
    from kv_cache_decode_quest_gb300 import synth
    W = synth.workloads()
    out = {}

    def quest_query(w, k, v, q, b, s):
        G = w.num_q_heads // w.num_kv_heads
        L = w.ctx[b] + s + 1
        for h in range(w.num_kv_heads):
            K, V = oracle.widen(k[h, :L]), oracle.widen(v[h, :L])
            qg = oracle.widen(q[s, b, h * G:(h + 1) * G])
            U = oracle.quest_bound(qg, *oracle.page_minmax(K))
            pages = oracle.quest_select(U, oracle.quest_k_pages(min(w.budget[b], 2 ** 31 - 1)))
            oracle.attend(qg, K[selected_tokens(pages, L)], V[selected_tokens(pages, L)],
                          1 / math.sqrt(w.head_dim))

    for name in ("tiny_quest", "quest_32k"):
        w = W[name]
        k, v = synth.quest_sequence(w, 0)
        q = synth.quest_queries(w)
        r, n = _timed_calls(lambda: quest_query(w, k, v, q, 0, 0), seconds)
        out[name] = {"queries_per_s": round(r, 3), "queries": n}
    w = W["ragged_quest_128k"]
    seqs = {b: synth.quest_sequence(w, b) for b in (0, 1)}      # one dense, one sparse request
    q = synth.quest_queries(w)
    cyc = [0]

    def ragged_query():
        b = cyc[0] % 2
        cyc[0] += 1
        quest_query(w, *seqs[b], q, b, 0)
    r, n = _timed_calls(ragged_query, seconds)
    out["ragged_quest_128k"] = {"queries_per_s": round(r, 4), "queries": n,
                                "sample": "alternating a full-budget and a 4096-budget request"}
    # SnapKV: one (request, KV head) compaction, and one decode query
    w = synth.scaled(W["snapkv_32k"], batch=1)
    inp = synth.snapkv_inputs(w, 0)
    G = w.num_q_heads // w.num_kv_heads
    scale = 1 / math.sqrt(w.head_dim)

    def compact_unit():
        K, V = oracle.widen(inp["k"][0][0]), oracle.widen(inp["v"][0][0])
        A = oracle.window_scores(oracle.widen(inp["q_win"][0][:, :G]), K, scale)
        keep = oracle.keep_positions(A, w.ctx, w.window, w.keep, w.pool_kernel)
        oracle.compact(K, V, keep)
    r, n = _timed_calls(compact_unit, seconds)
    units = W["snapkv_32k"].batch * w.num_kv_heads
    out["snapkv_32k_compaction"] = {"batches_per_s": round(r / units, 5), "units_timed": n,
                                    "sample": f"one (request, KV head) of the 8 x 32K batch, "
                                              f"rate divided by its {units} units"}
    kept = w.keep + w.window
    K, V = oracle.widen(inp["k"][0][0][:kept]), oracle.widen(inp["v"][0][0][:kept])
    qd = oracle.widen(inp["q_win"][0][0, :G])

    def snap_decode():
        for _ in range(w.num_kv_heads):
            oracle.attend(qd, K, V, scale)
    r, n = _timed_calls(snap_decode, seconds)
    out["snapkv_32k_decode"] = {"queries_per_s": round(r, 3), "queries": n,
                                "sample": f"{kept}-token attention per KV head"}
    # H2O: one decode step of one request over its 4 KV heads
    w = synth.scaled(W["h2o_16k"], batch=1)
    hi = synth.h2o_inputs(w)
    G = w.num_q_heads // w.num_kv_heads
    scale = 1 / math.sqrt(w.head_dim)
    st = oracle.h2o_init(oracle.widen(hi["q_win"][0][:, :G]), oracle.widen(hi["k"][0][0]),
                         oracle.widen(hi["v"][0][0]), w.budget, w.recent, scale)
    qn = oracle.widen(hi["q"][0, 0, :G])
    kn, vn = oracle.widen(hi["k_new"][0, 0, 0]), oracle.widen(hi["v_new"][0, 0, 0])

    def h2o_query():
        for _ in range(w.num_kv_heads):
            oracle.h2o_step(st, qn, kn, vn, w.ctx, w.budget, w.recent, scale)
    r, n = _timed_calls(h2o_query, seconds)
    out["h2o_16k"] = {"queries_per_s": round(r, 3), "queries": n}
    # cross-layer reuse: one request through 4 layers
    w = W["omnikv_32k"]
    lay = [synth.quest_sequence(w.layer(x), 0) for x in range(w.layers)]
    lq = [synth.quest_queries(w.layer(x)) for x in range(w.layers)]
    G = w.num_q_heads // w.num_kv_heads
    L = w.ctx[0] + 1

    def omni_query():
        for h in range(w.num_kv_heads):
            oracle.omnikv_layers([oracle.widen(lq[x][0, 0, h * G:(h + 1) * G]) for x in range(w.layers)],
                                 [oracle.widen(lay[x][0][h, :L]) for x in range(w.layers)],
                                 [oracle.widen(lay[x][1][h, :L]) for x in range(w.layers)],
                                 w.filters, w.budget[0], 1 / math.sqrt(w.head_dim))
    r, n = _timed_calls(omni_query, seconds)
    out["omnikv_32k"] = {"layer_queries_per_s": round(r * w.layers, 3), "queries": n}
    return out


def oracle_rates(seconds=2.0):
    """Single-threaded oracle rates per workload, in one spawned process."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(1) as pool:
        res = pool.apply(_oracle_rates_worker, (seconds,))
        pool.close()
        pool.join()
    return res


def cpu_baseline(name, seconds=12.0, cores=None, single=None):
    import multiprocessing as mp
    cores = cores or max(1, os.cpu_count() or 1)
    from kv_cache_decode_quest_gb300 import synth
    B = synth.workloads()[name].batch
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(name, i % B, seconds) for i in range(cores)])
        pool.close()
        pool.join()
    wall = time.perf_counter() - t0
    q = sum(r[0] for r in res)
    per_worker = [r[0] / r[1] for r in res]
    line = {"value": sum(per_worker), "unit": "queries/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"{q} oracle queries ({name}: page summaries, bound, top-k, fp64 "
                      f"attention per KV head), ~{seconds:.0f} s per core on {cores} "
                      f"single-threaded spawned workers, wall {wall:.1f} s"}
    if single is not None:
        line["single_core"] = {"value": single, "unit": "queries/s", "cores": 1}
    return line


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------

class QuestBench:
    """Drives a QuestRun through timed steps, wrapping around its step inputs
    (restoring the page summaries and lengths, outside the timed region)."""

    def __init__(self, name, device, mode="step", step_tuning=None):
        import torch
        from kv_cache_decode_quest_gb300 import synth, workloads
        self.torch = torch
        self.name = name
        self.mode = mode
        self.w = synth.workloads()[name]
        inputs = synth.quest_inputs(self.w)
        self.run = workloads.QuestRun(self.w, inputs, device=device, mode=mode,
                                      step_tuning=step_tuning)
        del inputs
        self.meta0 = self.run.kv.meta.clone()
        self.ctx0 = self.run.kv.ctx_len.clone()
        self.s = 0
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def next_index(self):
        if self.s == self.w.steps:
            self.run.kv.meta.copy_(self.meta0)
            self.run.kv.ctx_len.copy_(self.ctx0)
            self.s = 0
        s = self.s
        self.s += 1
        return s

    def bytes_for(self, s):
        import numpy as np
        ctx_now = np.asarray(self.w.ctx) + s + 1
        return self.run.algorithmic_bytes(ctx_now)

    def kernel_bytes(self, s):
        """Algorithmic bytes of the timed kernel: the whole step for the
        one-kernel step; K/V of the selected tokens, q and the output for the
        decode kernel."""
        b = self.bytes_for(s)
        return b["total"] if self.mode == "step" else b["kv"] + b["small"]

    def launches_per_step(self):
        return 1 if self.mode == "step" else 3   # score, top-k (+ append), decode

    def capture(self):
        """One CUDA graph per step index (the step's kernels); replaying graph s
        runs step s without host launch overhead."""
        torch = self.torch
        s0 = self.next_index()                    # warm-up eager step, then rewind
        self.run.step(s0)
        torch.cuda.synchronize()
        self.run.kv.meta.copy_(self.meta0)
        self.run.kv.ctx_len.copy_(self.ctx0)
        self.s = 0
        side = torch.cuda.Stream()
        self.graphs = []
        for s in range(self.w.steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self.run.step(s)
            self.graphs.append(g)
        torch.cuda.synchronize()

    def capture_kernel_timing(self):
        """A second graph per step index, the dominant kernel (the step kernel,
        or the decode kernel of the two-call step) bracketed by event nodes:
        replaying it times the kernel as the step graphs run it (no host
        launch latency inside the interval)."""
        torch = self.torch
        side = torch.cuda.Stream()
        self.kgraphs, self.kevents = [], []
        for s in range(self.w.steps):
            b = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            b.record()                            # torch creates the events on first record
            e.record()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self.run.step(s, ev_begin=b, ev_end=e)
            self.kgraphs.append(g)
            self.kevents.append((b, e))
        torch.cuda.synchronize()

    def timed_kernel(self, K, W):
        """Dominant kernel durations over K replays of the event-bracketed step
        graphs (L2 flushed before each), after W untimed ones."""
        torch = self.torch
        for _ in range(W):
            s = self.next_index()
            self.flush.zero_()
            self.kgraphs[s].replay()
        torch.cuda.synchronize()
        kern_ms, idx = [], []
        for _ in range(K):
            s = self.next_index()
            self.flush.zero_()
            self.kgraphs[s].replay()
            torch.cuda.synchronize()              # graph s's events are read before any re-use
            b, e = self.kevents[s]
            kern_ms.append(b.elapsed_time(e))
            idx.append(s)
        return kern_ms, idx

    def timed(self, K, W, graphs=True):
        """Step times (graph replay, or eager calls when graphs=False) and, in
        eager mode, the decode kernel's own time from events the library
        records around it."""
        torch = self.torch
        for _ in range(W):
            s = self.next_index()
            self.flush.zero_()
            if graphs:
                self.graphs[s].replay()
            else:
                self.run.step(s)
        torch.cuda.synchronize()
        E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        evs, idx = [], []
        for _ in range(K):
            s = self.next_index()
            self.flush.zero_()
            e = (E(), E(), E(), E())
            if graphs:
                e[0].record()
                self.graphs[s].replay()
                e[1].record()
            else:
                # torch creates an event on its first record(); the library then
                # re-records the kernel events around the decode kernel itself
                e[2].record()
                e[3].record()
                e[0].record()
                self.run.step(s, ev_begin=e[2], ev_end=e[3])
                e[1].record()
            evs.append(e)
            idx.append(s)
        torch.cuda.synchronize()
        step_ms = [e[0].elapsed_time(e[1]) for e in evs]
        kern_ms = None if graphs else [e[2].elapsed_time(e[3]) for e in evs]
        return step_ms, kern_ms, idx

    def timed_e2e(self, K, W):
        """Same steps through host buffers, as a serving loop runs them: each
        step's graph copies the NEXT step's q/k/v in (one row of pinned host
        memory) and the PREVIOUS step's output out (pinned host memory) on a
        second stream while the step's kernels run, the outputs double-buffered
        on the device.  Every timed step moves one step's inputs in and one
        step's result out."""
        torch = self.torch
        r = self.run
        S = r.S
        inh = r.step_inputs.cpu().pin_memory()
        oh = torch.empty((S,) + tuple(r.out.shape), dtype=r.out.dtype).pin_memory()
        outs = [torch.empty_like(r.out) for _ in range(2)]
        lses = [torch.empty_like(r.lse) for _ in range(2)]
        copies = torch.cuda.Stream()

        def one(s):
            main = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(main)
            copies.wait_event(fork)
            with torch.cuda.stream(copies):
                r.step_inputs[(s + 1) % S].copy_(inh[(s + 1) % S], non_blocking=True)
                oh[(s - 1) % S].copy_(outs[(s - 1) % 2], non_blocking=True)
            r.step(s, out=outs[s % 2], lse=lses[s % 2])
            join = torch.cuda.Event()
            join.record(copies)
            main.wait_event(join)

        self.run.kv.meta.copy_(self.meta0)
        self.run.kv.ctx_len.copy_(self.ctx0)
        r.step_inputs[0].copy_(inh[0])
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        graphs = []
        for s in range(S):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                one(s)
            graphs.append(g)
        torch.cuda.synchronize()
        self.s = 0
        for _ in range(W):
            s = self.next_index()
            self.flush.zero_()
            graphs[s].replay()
        torch.cuda.synchronize()
        evs = []
        for _ in range(K):
            s = self.next_index()
            self.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graphs[s].replay()
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
        h2d = inh[0].numel() * inh.element_size()
        d2h = oh[0].numel() * oh.element_size()
        return ms, h2d, d2h


def reduce_max(x, ws):
    """Max of x over the ranks (the timed region ends when the slowest replica does)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(per_rank_batch, steps, total_ms, ws):
    """Whole-job queries/s: every rank ran its own batch for `steps` steps; the
    job took the slowest rank's time."""
    return ws * per_rank_batch * steps / (total_ms / 1e3)


def barrier(ws):
    import torch
    cuda = torch.cuda.is_available()
    if cuda:
        torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    import __graft_entry__
    __graft_entry__.build()

    peak, peak_kind = peaks()
    qb = QuestBench(HEADLINE, device, mode=HEADLINE_MODE)
    B = qb.w.batch
    qb.capture()
    barrier(ws)
    with ClockSampler(local) as clk:
        step_ms, _, idx = qb.timed(args.steps, args.warmup, graphs=True)
    barrier(ws)
    total_ms = reduce_max(sum(step_ms), ws)
    ms_per_step = total_ms / args.steps
    value = replica_value(B, args.steps, total_ms, ws)
    bytes_steps = [qb.bytes_for(s) for s in idx]
    step_gbs = sum(b["total"] for b in bytes_steps) / (sum(step_ms) / 1e3) / 1e9

    # the dominant kernel's own duration: event nodes around it in replayed step graphs
    qb.capture_kernel_timing()
    kern_ms, kidx = qb.timed_kernel(args.steps, args.warmup)
    dec_bytes = [qb.kernel_bytes(s) for s in kidx]
    achieved = sum(dec_bytes) / (sum(kern_ms) / 1e3) / 1e9

    e2e_ms, h2d, d2h = qb.timed_e2e(args.steps, args.warmup)
    e2e_total = reduce_max(sum(e2e_ms), ws)
    e2e_value = replica_value(B, args.steps, e2e_total, ws)

    extra = {}
    if args.extras:
        extra = run_extras(args, device, peak)

    # oracle baselines last (spawned workers on the host cores, rank 0 only),
    # so that no GPU timing, the end-to-end one above all, runs on a host
    # that the workers still load: every workload's single-threaded oracle
    # rate, then the headline's on all host cores
    rates = oracle_rates(args.oracle_seconds) if (rank == 0 and args.oracle_seconds > 0) else {}
    cpu = (cpu_baseline(HEADLINE, seconds=args.cpu_seconds,
                        single=rates.get(HEADLINE, {}).get("queries_per_s"))
           if (rank == 0 and args.cpu_seconds > 0) else None)
    for key, val in extra.items():
        if key in rates:
            val["oracle_single_core"] = rates[key]

    if rank != 0:
        return
    kname, ksrc, krec = KERNEL_OF_MODE[HEADLINE_MODE]
    traffic = profiled_traffic(krec.format(HEADLINE), ksrc)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "queries/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "quest_32k: Qwen3-30B-A3B-shaped layer (32 q / 4 kv heads, "
                               "head_dim 128), batch 16, context 32768 + 1 token/step, page 16, "
                               "Quest budget 2048 tokens per KV head, K with 4 outlier channels x8",
                   "global_batch": B * ws, "seq_len": 32768, "parallelism": f"replicas x{ws}",
                   "l2": "flushed (512 MiB write) before every timed step",
                   "step": ("token append, Quest page scoring, per-KV-head top-k, view and "
                            "split-K decode + LSE merge in one persistent kernel (se_quest_step)"
                            if HEADLINE_MODE == "step" else
                            "Quest select with the token append fused (score, top-k + append, "
                            "view) + split-K decode + merge"),
                   "launch": "one CUDA graph per step index, replayed"},
        "roofline": {"bound": "hbm", "kernel": kname,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": int(sum(dec_bytes) / len(dec_bytes)),
                     "kernel_ms_per_launch": round(sum(kern_ms) / len(kern_ms), 5),
                     "kernel_timing": f"CUDA event nodes around {kname} inside the "
                                      "replayed step graphs, L2 flushed before each",
                     "step_algorithmic_gbs": round(step_gbs, 1),
                     "step_frac": round(step_gbs / peak, 4)},
        "e2e": {"value": round(e2e_value, 1), "unit": "queries/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "pinned host rows; each step's graph copies the next step's q/k/v in and "
                          "the previous step's output out on a second stream during its kernels "
                          "(outputs double-buffered on the device)"},
        "gpu_launches": qb.launches_per_step() * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if extra:
        line["extra"] = extra
    print(json.dumps(line), flush=True)


def timed_steps(step, K, W, flush, before=None):
    """W untimed then K timed calls of step(i, ev_begin, ev_end); the L2 is
    flushed before each.  Returns (step ms list, kernel ms list or None)."""
    import torch
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for i in range(W):
        if before:
            before(i)
        flush.zero_()
        step(i, None, None)
    torch.cuda.synchronize()
    evs = []
    for i in range(W, W + K):
        if before:
            before(i)
        flush.zero_()
        e = (E(), E(), E(), E())
        e[2].record()
        e[3].record()
        e[0].record()
        step(i, e[2], e[3])
        e[1].record()
        evs.append(e)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b, _, _ in evs], [c.elapsed_time(d) for _, _, c, d in evs]


EXTRAS = ("tiny_quest", "ragged_quest_128k", "omnikv_32k", "snapkv_32k", "h2o_16k")


def run_extras(args, device, peak, only=None):
    """The other workloads of the path, timed the same way (reported beside the headline)."""
    import torch
    out = {}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    want = set(EXTRAS if only is None else [only])
    if "tiny_quest" in want:
        tiny(out, device)
    # ragged 64K-128K Quest decode (half dense-equivalent), split-K up to 64
    if "ragged_quest_128k" in want:
        ragged(out, device, peak)
    if "omnikv_32k" in want:
        omnikv(out, device, peak, flush)
    if "snapkv_32k" in want:
        snapkv(out, device, peak, flush)
    if "h2o_16k" in want:
        h2o(out, device, peak, flush)
    return out


def ragged(out, device, peak):
    import torch
    qb = QuestBench("ragged_quest_128k", device, mode=RAGGED_MODE)
    K = min(16, qb.w.steps)
    qb.capture()
    step_ms, _, idx = qb.timed(K, 3, graphs=True)
    qb.capture_kernel_timing()
    kern_ms, kidx = qb.timed_kernel(K, 3)
    bytes_steps = [qb.bytes_for(s) for s in idx]
    dec = sum(qb.kernel_bytes(s) for s in kidx)
    out["ragged_quest_128k"] = {
        "queries_per_s": round(qb.w.batch * K / (sum(step_ms) / 1e3), 1),
        "ms_per_step": round(sum(step_ms) / K, 5),
        "kernel": KERNEL_OF_MODE[RAGGED_MODE][0],
        "kernel_gbs": round(dec / (sum(kern_ms) / 1e3) / 1e9, 1),
        "kernel_frac": round(dec / (sum(kern_ms) / 1e3) / 1e9 / peak, 4),
        "step_gbs": round(sum(b["total"] for b in bytes_steps) / (sum(step_ms) / 1e3) / 1e9, 1),
        "steps": K, "warmup": 3}
    del qb
    torch.cuda.empty_cache()


def tiny(out, device):
    """The one-sequence, one-query Quest step (2K context, 8 of 128 pages): a
    latency figure (no roofline target), one replayed graph per step."""
    import torch
    qb = QuestBench("tiny_quest", device, mode=TINY_MODE)
    qb.capture()
    step_ms, _, _ = qb.timed(50, 5, graphs=True)
    out["tiny_quest"] = {
        "us_per_step": round(sum(step_ms) / len(step_ms) * 1e3, 2),
        "us_per_step_min": round(min(step_ms) * 1e3, 2),
        "queries_per_s": round(len(step_ms) / (sum(step_ms) / 1e3), 1),
        "step": ("Quest select with the append fused + split-K decode, one replayed graph"
                 if TINY_MODE == "fused" else
                 "the whole step in one kernel (se_quest_step), one replayed graph"),
        "steps": 50, "warmup": 5}
    del qb
    torch.cuda.empty_cache()


def omnikv(out, device, peak, flush):
    """Cross-layer selection reuse: 16 x 32K requests through 4 attention
    layers, layer 0 selecting with Quest and layers 1-3 decoding through its
    view; one replayed graph per step index, L2 flushed before each step."""
    import numpy as np
    import torch
    from kv_cache_decode_quest_gb300 import synth, workloads
    w = synth.workloads()["omnikv_32k"]
    run = workloads.OmniRun(w, synth.omnikv_inputs(w), device=device)
    side = torch.cuda.Stream()
    graphs = []
    for s in range(w.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            run.step(s)
        graphs.append(g)
    torch.cuda.synchronize()
    W, K = 3, w.steps - 3
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for s in range(W):
        flush.zero_()
        graphs[s].replay()
    evs = []
    for s in range(W, W + K):
        flush.zero_()
        e = (E(), E())
        e[0].record()
        graphs[s].replay()
        e[1].record()
        evs.append(e)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    nbytes = sum(run.algorithmic_bytes(np.asarray(w.ctx) + s + 1)["total"] for s in range(W, W + K))
    gbs = nbytes / (sum(ms) / 1e3) / 1e9
    out["omnikv_32k"] = {
        "layer_queries_per_s": round(w.batch * w.layers * K / (sum(ms) / 1e3), 1),
        "steps_per_s": round(K / (sum(ms) / 1e3), 1),
        "ms_per_step": round(sum(ms) / K, 5),
        "step_algorithmic_gbs": round(gbs, 1), "step_frac": round(gbs / peak, 4),
        "layers": w.layers, "filter_layers": list(w.filters), "batch": w.batch,
        "status": run.status(), "steps": K, "warmup": W}
    del run, graphs
    torch.cuda.empty_cache()


def snapkv(out, device, peak, flush):
    """SnapKV: compaction of a batch of 8 x 32K prefills, then decode of the
    64 compacted requests (8 seeded compaction batches)."""
    import torch
    from kv_cache_decode_quest_gb300 import binding as se
    from kv_cache_decode_quest_gb300 import synth, workloads
    w = synth.workloads()["snapkv_32k"]
    sr = workloads.SnapKVRun(w, device=device)
    scratch = se.VarlenKV.empty(w.batch, w.num_kv_heads, sr.seg_cap, w.head_dim, device=device)

    def compact(i, e0, e1):
        if e0 is not None:
            e0.record()
        se.se_snapkv_compact(sr.prefill, sr.q_win, w.batch, w.num_q_heads, w.window,
                             w.pool_kernel, w.keep, w.window, sr.scale, scratch, sr.ws_snap)
        if e1 is not None:
            e1.record()
    c_ms, _ = timed_steps(compact, 5, 3, flush)
    Bh = w.batch * w.num_kv_heads
    L, D, G = w.ctx, w.head_dim, w.num_q_heads // w.num_kv_heads
    kept = min(w.keep, L - w.window) + w.window
    c_bytes = Bh * (L * D * 2 + 2 * kept * D * 2 * 2)       # K read once, kept K/V read + written
    c_flops = 2 * 2 * Bh * w.window * G * L * D              # two passes of S = Q K^T
    c_s = sum(c_ms) / len(c_ms) / 1e3
    tf_peak, sm_mhz, tf_kind = tensor_peak()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    ex2 = 2 * Bh * w.window * G * L                           # one exp2 per (row, key) per pass
    ex2_peak = EX2_PER_CLOCK_PER_SM * sms * sm_mhz * 1e6
    out["snapkv_32k_compaction"] = {
        "ms_per_batch": round(c_s * 1e3, 4),
        "prefill_tokens_per_s": round(w.batch * L / c_s, 1),
        "algorithmic_gbs": round(c_bytes / c_s / 1e9, 1),
        "tensor_tflops": round(c_flops / c_s / 1e12, 1),
        "roofs": {
            "hbm_frac": round(c_bytes / c_s / 1e9 / peak, 4),
            "tensor_frac": round(c_flops / c_s / 1e12 / tf_peak, 4),
            "tensor_peak_tflops": tf_peak, "tensor_peak_kind": tf_kind + " bf16 burst",
            "ex2_per_s": round(ex2 / c_s, 1),
            "ex2_frac": round(ex2 / c_s / ex2_peak, 4),
            "ex2_peak_per_s": round(ex2_peak, 1),
            "ex2_peak": f"{EX2_PER_CLOCK_PER_SM} per clock per SM x {sms} SMs x {sm_mhz:.0f} MHz",
            "scope": "whole compaction call (both scoring passes, pool + top-k, gather)"},
        "batch": w.batch, "ctx": L}
    K2 = min(32, w.steps - 3)
    s_ms, s_k = timed_steps(lambda i, a, b: sr.step(i, a, b), K2, 3, flush)
    units_s = sr.Bt * w.num_kv_heads
    # timed step j attends kept + 3 (warm-up appends) + j + 1 tokens per unit
    kv_b = sum(units_s * (kept + 4 + j) * 2 * D * 2 for j in range(K2)) / K2
    out["snapkv_32k_decode"] = {
        "queries_per_s": round(sr.Bt * K2 / (sum(s_ms) / 1e3), 1),
        "ms_per_step": round(sum(s_ms) / K2, 5),
        "decode_gbs": round(kv_b / (sum(s_k) / len(s_k) / 1e3) / 1e9, 1),
        "decode_frac": round(kv_b / (sum(s_k) / len(s_k) / 1e3) / 1e9 / peak, 4),
        "batch": sr.Bt, "steps": K2, "warmup": 3}
    del sr, scratch
    torch.cuda.empty_cache()


def h2o(out, device, peak, flush):
    """H2O: 64 requests, 4096 retained of 16K, one eviction per unit per step."""
    import torch
    from kv_cache_decode_quest_gb300 import synth, workloads
    w = synth.workloads()["h2o_16k"]
    hr = workloads.H2ORun(w, device=device)
    K3 = min(64, w.steps - 3)
    h_ms, _ = timed_steps(lambda i, a, b: hr.step(i), K3, 3, flush)
    units = w.batch * w.num_kv_heads
    n = w.budget + 1
    G = w.num_q_heads // w.num_kv_heads
    h_bytes = units * (n * 2 * w.head_dim * 2 + n * G * 4 * 2 + n * 4 * 2)
    out["h2o_16k"] = {
        "queries_per_s": round(w.batch * K3 / (sum(h_ms) / 1e3), 1),
        "ms_per_step": round(sum(h_ms) / K3, 5),
        "step_algorithmic_gbs": round(h_bytes / (sum(h_ms) / K3 / 1e3) / 1e9, 1),
        "step_frac": round(h_bytes / (sum(h_ms) / K3 / 1e3) / 1e9 / peak, 4),
        "batch": w.batch, "steps": K3, "warmup": 3}
    del hr
    torch.cuda.empty_cache()


def run_only(args):
    import torch
    torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    peak, _ = peaks()
    res = run_extras(args, "cuda:0", peak, only=args.only)
    print(json.dumps({"only": args.only, **res}), flush=True)


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is one query of
    the headline workload (rank 0 only)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    import oracle
    from kv_cache_decode_quest_gb300 import synth
    w = synth.workloads()[HEADLINE]
    G = w.num_q_heads // w.num_kv_heads
    scale = 1.0 / math.sqrt(w.head_dim)
    seqs = {}

    def query(i):
        b, s = i % w.batch, (i // w.batch) % w.steps
        if b not in seqs:
            seqs.clear()
            seqs[b] = synth.quest_sequence(w, b)
        k, v = seqs[b]
        L = w.ctx[b] + s + 1
        for h in range(w.num_kv_heads):
            K = oracle.widen(k[h, :L])
            V = oracle.widen(v[h, :L])
            qg = oracle.widen(q[s, b, h * G:(h + 1) * G])
            U = oracle.quest_bound(qg, *oracle.page_minmax(K))
            pages = oracle.quest_select(U, oracle.quest_k_pages(w.budget[b]))
            tok = oracle.quest.selected_tokens(pages, L)
            oracle.attend(qg, K[tok], V[tok], scale)

    q = synth.quest_queries(w)
    # order queries so a sequence's inputs are generated once per run of steps
    order = [b + w.batch * s for b in range(w.batch) for s in range(w.steps)]
    for i in range(args.warmup):
        query(order[i % len(order)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        query(order[(args.warmup + i) % len(order)])
    dt = time.perf_counter() - t0
    value = args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "queries/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "global_batch": w.batch, "seq_len": 32768,
                   "parallelism": "none (host CPU)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "queries/s", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{args.steps} oracle queries of {HEADLINE} (one sequence's "
                                   f"decode step over 4 KV heads each), single thread"},
        "e2e": {"value": round(value, 3), "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="seconds of oracle work per host core for cpu_baseline (0 = skip)")
    ap.add_argument("--oracle-seconds", type=float, default=2.0,
                    help="seconds of single-threaded oracle work per workload (0 = skip)")
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    ap.add_argument("--only", choices=EXTRAS, default=None,
                    help="run one of the other workloads alone and print its figures")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
