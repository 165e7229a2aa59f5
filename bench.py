"""Benchmark: draft+verify attention steps/s of the TriForce decode step at 128K.

One step = for every layer, in order: chunk scores + top-k + sparse decode
attention over the retrieved chunks (the Force 2 retrieval drafter, one fused
launch; --two-call-draft runs it as the separate top-k and sparse-attention
calls), then full-cache verification of gamma+1 = 6 queries (Force 3)
with the sink + window attention of the decode queries (Force 1) computed as
extra query rows of the same launch (tf_verify_window_attn).
Workload: the full 32-layer Llama2-7B-128K KV cache (32 heads x 128 dims x
131072 tokens, bf16, 64 GiB), seeded synthetic data with 1% planted chunks.
Consecutive steps take different seeded queries (four sets per layer, cycled),
and the retrieval drafter gets 0.7 x the previous step's cut of each layer as
a lower bound on this step's cut (it changes only the time); "cold_start" is
the same step without the bound.
After it, in the same run, the same step on the GQA batch (Llama-3-8B style,
batch 4, 32/8 heads, 128K, 32 layers) and on the mixed batch (batch 8,
contexts 16K..128K, 32/8 heads, 16 layers), each reported under "workloads".

Default (impl=triforce): the CUDA library, inputs resident in HBM; prints one
JSON line with steps/s, the verify kernel's roofline, an end-to-end number
(queries copied from pinned host memory and outputs copied back inside the
timed region) and the float64 oracle timed on every host core (one
single-threaded worker process per core) on a bounded sample of the workload.
impl=reference: the oracle alone, on the same pool, one bounded sample per step.

Multi-GPU (torchrun): each rank runs an independent replica of the step on its
own GPU (the path has no exchange step); value = all ranks' steps / max time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "draft+verify attn steps/s at 128K (Llama2-7B shape); achieved HBM GB/s vs peak"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="triforce", choices=["triforce", "reference"])
    ap.add_argument("--workload", default="llama2-7b-128k-32layer")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling runs only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capture the step (every layer's launches) once as a CUDA graph and replay it")
    ap.add_argument("--two-call-draft", action="store_true",
                    help="run the retrieval drafter as tf_chunk_scores_topk + tf_sparse_decode_attn")
    ap.add_argument("--extra-workloads", default="llama3-8b-gqa-128k-b4,mixed-b8-gqa-16k-128k",
                    help="comma-separated workloads timed after the headline one ('none': skip)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers


def dist_setup(n_gpus):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Largest value over all ranks (the slowest replica sets the job time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(steps, elapsed_local_s, world, device="cuda"):
    """Whole-job steps/s: every rank runs `steps` steps of its own replica; the
    job ends when the slowest rank does.  Returns (steps/s, max elapsed)."""
    el = max_over_ranks(elapsed_local_s, world, device)
    return world * steps / el, el


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_hash(name):
    path = os.path.join(ROOT, "hierarchical_speculative_decoding_gb300", "csrc", name)
    h = hashlib.sha256()
    with open(path, "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_file, workload):
    """DRAM bytes per launch of the kernel on this workload from the committed ncu
    summary, if it was taken on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel_file)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and parts[0] == kernel_file and parts[1] == want and parts[2] == workload:
                return float(parts[3])
    return None


# ---------------------------------------------------------------- CPU oracle (every host core)

_ORACLE_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
               "CUDA_VISIBLE_DEVICES": ""}


def _pool_warm(_):
    """Import the oracle and the input generators in a pool worker before any
    unit is timed (and hold the worker briefly so each gets one task)."""
    sys.path.insert(0, ROOT)
    import numpy  # noqa: F401
    import torch  # noqa: F401

    from hierarchical_speculative_decoding_gb300 import synth  # noqa: F401
    from oracle import triforce  # noqa: F401

    time.sleep(0.3)
    return os.getpid()


def cpu_unit_worker(w_name, unit, seed):
    """The float64 oracle on one (layer, KV head) unit of the workload at full
    context: scores + top-k, sparse decode, window and verify attention.
    Returns the seconds of oracle compute (input generation excluded)."""
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    from hierarchical_speculative_decoding_gb300 import synth
    from oracle import triforce as O

    w = synth.WORKLOADS[w_name]
    L = int(synth.seq_lens_for(w).max())
    unit_w = synth.Workload(w.name + "-unit", 1, w.G, 1, w.D, L, 1, w.chunk, w.budget, w.n_sink, w.window, w.T,
                            w.gamma, w.vocab, w.planted_frac, seed + unit)
    scale = w.D ** -0.5
    seq = synth.seq_lens_for(unit_w)
    q, Q = synth.decode_queries(unit_w, 0)
    K, V, _ = synth.kv_cache(unit_w, 0, q, seq)
    kb = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    qb, Qb, Kb, Vb, sl = kb(q), kb(Q), kb(K), kb(V), seq.numpy()
    M = O.build_chunk_means(Kb, sl, w.chunk)  # prefill-time index, not part of the step
    t0 = time.perf_counter()
    idx, nsel, *_ = O.chunk_scores_topk(qb, M, sl, L, w.chunk, w.kc, 1)
    O.sparse_decode_attn(qb, Kb, Vb, sl, idx, nsel, w.chunk, scale)
    O.stream_window_attn(qb, Kb, Vb, sl, w.n_sink, w.window, scale)
    O.verify_attn(Qb, Kb, Vb, sl, scale)
    return time.perf_counter() - t0


def cpu_baseline(w, units_per_worker=2):
    """The oracle, as it stands, on every host core: a spawn process pool (safe
    beside a CUDA context) with one single-threaded worker per core, each
    timing whole (layer, KV head) units at full context; all workers run at
    once, so the per-unit times include their contention.  Throughput =
    workers / mean unit time, scaled to one full step (units x layers)."""
    import concurrent.futures as cf
    import multiprocessing as mp

    workers = max(1, os.cpu_count() or 1)
    n_units = units_per_worker * workers
    saved = {k: os.environ.get(k) for k in _ORACLE_ENV}
    os.environ.update(_ORACLE_ENV)
    try:
        with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            list(ex.map(_pool_warm, range(workers)))
            t0 = time.perf_counter()
            times = list(ex.map(cpu_unit_worker, [w.name] * n_units, range(n_units), [7] * n_units))
            wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    per_unit = statistics.mean(times)
    units_per_step = w.B * w.Hkv * w.layers
    value = workers / per_unit / units_per_step
    return {"value": value, "unit": "steps/s", "cores": workers, "host_cpu_count": os.cpu_count(),
            "kind": "oracle", "threads_per_worker": 1,
            "sample": (f"{n_units} (layer, KV head) units at full context, float64 numpy oracle, {workers} "
                       f"single-threaded worker processes at once ({wall:.2f} s wall), {per_unit:.3f} s per unit; "
                       f"scaled by {units_per_step} units per step")}


# ---------------------------------------------------------------- GPU arm


def _ev():
    import torch

    return torch.cuda.Event(enable_timing=True)


_FLUSH = {}


def _median_call_ms(fn, stream, reps=5, warm=1, agg=statistics.median):
    """Median (or `agg`) device time of fn() on `stream`, each call bracketed
    by CUDA events behind a queued 512 MB memset: the memset keeps the GPU busy
    while the host enqueues the event, the call and the closing event (so host
    launch cost is not timed) and leaves L2 cold."""
    import torch

    if "buf" not in _FLUSH:
        _FLUSH["buf"] = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=torch.cuda.current_device())
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        _FLUSH["buf"].zero_()
        a, b = _ev(), _ev()
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return agg(out)


def graph_loop_ms(calls, stream, replays=5):
    """Per-call device time of a loop of short launches: the loop is captured
    once as a CUDA graph and replayed, so host launch cost (larger than these
    kernels through the Python binding) stays out of the measurement."""
    import torch

    for c in calls:  # first calls outside the capture (per-device set-up)
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    a, b = _ev(), _ev()
    a.record(stream)
    for _ in range(replays):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (replays * len(calls))
    del g
    return ms


def window_launches(G, T):
    """Launches tf_verify_window_attn makes for G query heads per KV head and T
    verify tokens: one when the G window rows fill padding rows of the verify
    kernel (no more 32-row groups, no wider group rounded up to 8 rows), else
    two (the library's rule; tests compare it with the workspace sizes)."""
    groups = lambda r: -(-r // 32)
    width = lambda r: -(-min(r, 32) // 8)
    fits = groups(G * (T + 1)) == groups(G * T) and width(G * (T + 1)) == width(G * T)
    return 1 if fits else 2


def window_in_draft(G, T):
    """Whether the step gives the window attention to the drafter: where the
    window rows would widen the verify launch (two launches), the fused draft
    carries them for two to four query heads per KV head
    (tf_retrieval_window_draft_attn), so a layer stays two launches."""
    return window_launches(G, T) == 2 and 2 <= G <= 4


N_QUERY_SETS = 4   # consecutive steps cycle through this many seeded query sets
HINT_SCALE = 0.7  # the draft's cut bound: the previous step's cut of the layer x 0.7


class StepState:
    """Resident inputs, outputs and workspaces of one workload's decode step.
    Consecutive steps take different seeded queries (N_QUERY_SETS sets per
    layer; set 0 is the one the planted chunks follow), so the retrieval
    drafter's cut moves from step to step and the previous step's cut is a
    bound, not the answer."""

    def __init__(self, w, layers, dev, tf, synth):
        import torch

        self.w, self.layers, self.dev = w, layers, dev
        B, Hq, Hkv, L, D, T = w.B, w.Hq, w.Hkv, w.L, w.D, w.T
        self.Cmax = -(-L // w.chunk)
        self.scale = D ** -0.5
        self.K = torch.empty((layers, B, Hkv, L, D), dtype=torch.bfloat16, device=dev)
        self.V = torch.empty_like(self.K)
        self.M = torch.empty((layers, B, Hkv, self.Cmax, D), dtype=torch.bfloat16, device=dev)
        self.seq_cpu = synth.seq_lens_for(w)
        self.seq = self.seq_cpu.to(dev)
        qs, Qs = [[] for _ in range(N_QUERY_SETS)], [[] for _ in range(N_QUERY_SETS)]
        for l in range(layers):
            for k in range(N_QUERY_SETS):
                q, Q = synth.decode_queries(w, l + 1000 * k, device=dev)
                qs[k].append(q)
                Qs[k].append(Q)
            synth.kv_cache(w, l, qs[0][l], self.seq_cpu, device=dev, K_out=self.K[l], V_out=self.V[l])
        self.q_sets = torch.stack([torch.stack(x) for x in qs])  # [sets, layers, B, Hq, D]
        self.Q_sets = torch.stack([torch.stack(x) for x in Qs])
        self.q = self.q_sets[0].clone()  # the live input buffers (host copies land here end to end)
        self.Q = self.Q_sets[0].clone()
        self.cut = torch.full((layers, B, Hkv), float("nan"), dtype=torch.float32, device=dev)
        self.hint = torch.full_like(self.cut, float("nan"))
        for l in range(layers):
            tf.tf_build_chunk_means(self.K[l], self.seq, self.M[l])
        self.idx = torch.empty((layers, B, Hkv, w.kc), dtype=torch.int32, device=dev)
        self.nsel = torch.empty((layers, B, Hkv), dtype=torch.int32, device=dev)
        self.o_sp = torch.empty((layers, B, Hq, D), dtype=torch.float32, device=dev)
        self.o_win = torch.empty((layers, B, Hq, D), dtype=torch.float32, device=dev)
        self.o_ver = torch.empty((layers, B, Hq, T, D), dtype=torch.float32, device=dev)
        self.ws_topk = tf.workspace(tf.tf_chunk_scores_topk_workspace(B, Hkv, L), dev)
        self.ws_sp = tf.workspace(tf.tf_sparse_decode_attn_workspace(B, Hq, Hkv, w.kc), dev)
        self.ws_win = tf.workspace(tf.tf_stream_window_attn_workspace(B, Hq, Hkv, w.n_sink, w.window), dev)
        self.ws_ver = tf.workspace(tf.tf_verify_attn_workspace(B, Hq, Hkv, L, T), dev)
        self.ws_vw = tf.workspace(tf.tf_verify_window_attn_workspace(B, Hq, Hkv, L, T, w.n_sink, w.window), dev)
        self.vw_launches = window_launches(Hq // Hkv, T)
        self.window_in_draft = window_in_draft(Hq // Hkv, T)
        torch.cuda.synchronize()

    def bytes_per_launch(self):
        """Algorithmic bytes of one layer's launches, from the actual lengths
        (and, for the drafter, the valid rows of the chunks it selected)."""
        import torch

        w = self.w
        B, Hq, Hkv, D, T = w.B, w.Hq, w.Hkv, w.D, w.T
        row = D * 2
        lens = [min(max(int(x), 0), w.L) for x in self.seq_cpu.tolist()]
        C = [-(-x // w.chunk) for x in lens]
        sel_rows = 0
        nsel = self.nsel[0].cpu()
        idx = self.idx[0].cpu()
        for b in range(B):
            for g in range(Hkv):
                ids = idx[b, g, : int(nsel[b, g])].to(torch.int64)
                sel_rows += int(torch.clamp(lens[b] - ids * w.chunk, 0, w.chunk).sum())
        q_io = B * Hq * D * (2 + 4)
        means = sum(Hkv * c * row for c in C)
        ids = B * Hkv * w.kc * 4
        return {
            "topk": means + B * Hq * D * 2 + ids,
            "sparse": 2 * sel_rows * row + ids + q_io,
            "draft": means + ids + 2 * sel_rows * row + q_io + (
                sum(2 * Hkv * min(x, w.n_sink + w.window) * row for x in lens) + B * Hq * D * 4
                if self.window_in_draft else 0),
            "window": sum(2 * Hkv * min(x, w.n_sink + w.window) * row for x in lens) + q_io,
            # in one launch the window rows read keys the verify rows read anyway: only their queries
            # and outputs add
            "verify": sum(2 * Hkv * x * row for x in lens) + B * Hq * T * D * (2 + 4) + (
                q_io if self.vw_launches == 1 else 0),
        }


def make_step(st, tf, two_call, stream, hinted=True, split_window=False):
    """One decode step over the layers.  step(evs, k) takes query set k (None:
    the live buffers st.q / st.Q).  With hinted, the fused drafter gets the
    previous step's cut of each layer x HINT_SCALE as a lower bound (a decode
    loop has it for free; one elementwise op per step forms it).  Window and
    verify: one tf_verify_window_attn call; with split_window, where that call
    makes two launches, the same two launches as two calls (an event between
    them for the per-kernel breakdown)."""
    import torch

    w = st.w
    wid = st.window_in_draft and not two_call  # the window attention in the drafter's launch
    split = split_window and st.vw_launches == 2 and not wid
    kinds = ("draft", "window", "verify") if split else ("draft", "verify")
    hinted = hinted and not two_call

    def draft(l, q=None):
        q = st.q if q is None else q
        if two_call:
            tf.tf_chunk_scores_topk(q[l], st.M[l], st.seq, w.L, w.kc, st.idx[l], st.nsel[l], ws=st.ws_topk)
            tf.tf_sparse_decode_attn(q[l], st.K[l], st.V[l], st.seq, st.idx[l], st.nsel[l], st.scale,
                                     out=st.o_sp[l], ws=st.ws_sp)
        elif wid:
            tf.tf_retrieval_window_draft_attn(q[l], st.M[l], st.K[l], st.V[l], st.seq, w.kc, st.scale, w.n_sink,
                                              w.window, idx=st.idx[l], n_sel=st.nsel[l], out=st.o_sp[l],
                                              wout=st.o_win[l], s_cut=st.cut[l],
                                              cut_hint=st.hint[l] if hinted else None)
        else:
            tf.tf_retrieval_draft_attn(q[l], st.M[l], st.K[l], st.V[l], st.seq, w.kc, st.scale, idx=st.idx[l],
                                       n_sel=st.nsel[l], out=st.o_sp[l], s_cut=st.cut[l],
                                       cut_hint=st.hint[l] if hinted else None)

    def step(evs=None, k=None, after=None):
        q = st.q if k is None else st.q_sets[k % N_QUERY_SETS]
        Q = st.Q if k is None else st.Q_sets[k % N_QUERY_SETS]
        if hinted:
            torch.mul(st.cut, HINT_SCALE, out=st.hint)
        for l in range(st.layers):
            if evs is not None:
                evs[l][0].record(stream)
            draft(l, q)
            if evs is not None:
                evs[l][1].record(stream)
            if split:
                tf.tf_stream_window_attn(q[l], st.K[l], st.V[l], st.seq, w.n_sink, w.window, st.scale,
                                         out=st.o_win[l], ws=st.ws_win)
                if evs is not None:
                    evs[l][2].record(stream)
                tf.tf_verify_attn(Q[l], st.K[l], st.V[l], st.seq, st.scale, out=st.o_ver[l], ws=st.ws_ver)
            elif wid:
                tf.tf_verify_attn(Q[l], st.K[l], st.V[l], st.seq, st.scale, out=st.o_ver[l], ws=st.ws_ver)
            else:
                tf.tf_verify_window_attn(Q[l], q[l], st.K[l], st.V[l], st.seq, w.n_sink, w.window, st.scale,
                                         out=st.o_ver[l], wout=st.o_win[l], ws=st.ws_vw)
            if evs is not None:
                evs[l][len(kinds)].record(stream)
            if after is not None:
                after(l)

    return step, draft, kinds


def e2e_graphs(st, step, q_host, Q_host, outs_host):
    """One CUDA graph per query set for the end-to-end loop: the step's queries
    are copied from pinned host memory first; each layer's outputs go back on a
    copy stream as soon as the layer is done, while the next layers run.  Every
    copy of the step is inside the graph, and the graph ends when the last one
    has landed.  (Waiting for each layer's queries separately cost more than
    it overlapped: the extra graph dependency in front of each layer's first
    launch stops it from starting early behind the previous launch.)"""
    import torch

    copy = torch.cuda.Stream()
    outs_dev = (st.o_sp, st.o_win, st.o_ver)
    graphs = []
    for k in range(N_QUERY_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cur = torch.cuda.current_stream()
            st.q.copy_(q_host[k], non_blocking=True)
            st.Q.copy_(Q_host[k], non_blocking=True)

            def after(l):
                done = torch.cuda.Event()
                done.record(cur)
                copy.wait_event(done)
                with torch.cuda.stream(copy):
                    for h, d in zip(outs_host, outs_dev):
                        h[l].copy_(d[l], non_blocking=True)

            step(None, None, after=after)
            join = torch.cuda.Event()
            join.record(copy)
            cur.wait_event(join)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


class StepCycle:
    """Calls step(k=0), step(k=1), ... : every call takes the next query set."""

    def __init__(self, step):
        self.step, self.k = step, 0

    def __call__(self, evs=None):
        self.step(evs, self.k)
        self.k += 1


def time_steps(run_step, steps, stream, world, local):
    """The headline region: a start and an end event only (events between
    kernels would stop programmatic dependent launch from overlapping them)."""
    import torch

    t_start, t_end = _ev(), _ev()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for _ in range(steps):
            run_step()
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    value, elapsed_s = job_throughput(steps, t_start.elapsed_time(t_end) / 1e3, world)
    return value, elapsed_s, clocks.summary()


def breakdown_cycle(st, tf, args, stream, k):
    """The step for the per-kernel breakdown (window and verify as separate
    calls where tf_verify_window_attn makes two launches), continuing at
    query set k.  Returns the cycle and its kinds."""
    step, _, kinds = make_step(st, tf, args.two_call_draft, stream, split_window=True)
    cyc = StepCycle(step)
    cyc.k = k
    return cyc, kinds


def verify_label(st):
    if st.vw_launches == 1:
        return "tf_verify_window_attn (one launch: the window rows inside the verify launch)"
    if st.window_in_draft:
        return "tf_verify_attn (the window attention rides in the drafter's launch)"
    return "tf_verify_attn, after tf_stream_window_attn (the two launches tf_verify_window_attn makes here)"


def draft_label(st, two_call):
    if two_call:
        return "tf_chunk_scores_topk + tf_sparse_decode_attn"
    if st.window_in_draft:
        return "tf_retrieval_window_draft_attn (scores, top-k, sparse and window attention in one launch)"
    return "tf_retrieval_draft_attn"


def launches_per_layer(st, two_call):
    if two_call:
        return 2 + st.vw_launches
    return 2 if st.window_in_draft else 1 + st.vw_launches


def per_kernel_times(step, layers, k_steps, kinds):
    """A second region with an event before and after every launch (step: a
    StepCycle, so these steps too take new queries)."""
    import torch

    evs = [[[_ev() for _ in range(len(kinds) + 1)] for _ in range(layers)] for _ in range(k_steps)]
    torch.cuda.synchronize()
    for s in range(k_steps):
        step(evs[s])
    torch.cuda.synchronize()
    per_kind = {k: [] for k in kinds}
    for s in range(k_steps):
        for l in range(layers):
            for i, k in enumerate(kinds):
                per_kind[k].append(evs[s][l][i].elapsed_time(evs[s][l][i + 1]))
    return per_kind


def kernel_entry(nbytes, ms, peak):
    gbps = nbytes / (ms / 1e3) / 1e9
    return {"ms": round(ms, 5), "GBps": round(gbps, 1), "frac_hbm": round(gbps / peak, 4)}


def measure_level1(st, w, tf, dev, stream, peak):
    """Level-1 verification over the retrieval cache (not part of the step):
    the step's selection, T verify queries, back-to-back calls over the layers
    replayed as one CUDA graph; and its fixed cost, the same calls over the
    first 16 selected chunks."""
    import torch

    B, Hq, Hkv, D, T = w.B, w.Hq, w.Hkv, w.D, w.T
    ws_sv = tf.workspace(tf.tf_sparse_verify_attn_workspace(B, Hq, Hkv, w.kc, T), dev)
    o_sv = torch.empty((B, Hq, T, D), dtype=torch.float32, device=dev)

    def sv_calls(idx_all, nsel_all):
        return [lambda l=l: tf.tf_sparse_verify_attn(st.Q[l], st.K[l], st.V[l], st.seq, idx_all[l], nsel_all[l],
                                                     st.scale, out=o_sv, ws=ws_sv) for l in range(st.layers)]

    sv_ms = graph_loop_ms(sv_calls(st.idx, st.nsel), stream)
    # selected chunks (clipped to each context) and the candidate rows, K and V
    rows = sum(min(w.kc * w.chunk, max(int(n), 0)) + T for n in st.seq_cpu.tolist())
    sv_bytes = 2 * Hkv * rows * D * 2 + B * Hq * T * D * (2 + 4)
    out = dict(kernel_entry(sv_bytes, sv_ms, peak), calls="tf_sparse_verify_attn",
               timing="back to back over the layers, replayed as one CUDA graph")
    idx16 = torch.full_like(st.idx, -1)
    idx16[:, :, :, :16] = st.idx[:, :, :, :16]
    nsel16 = torch.clamp(st.nsel, max=16)
    out["floor_kc16_us"] = round(graph_loop_ms(sv_calls(idx16, nsel16), stream) * 1e3, 2)
    return out


def draft_back_to_back_ms(st, draft, cyc, stream):
    """The retrieval draft alone, back to back over the layers, on the next
    query set (with the bounds the last step left): consecutive launches
    overlap through programmatic dependent launch (no events between them),
    and every layer's means and K/V are cold."""
    import torch

    q = st.q_sets[cyc.k % N_QUERY_SETS]
    torch.mul(st.cut, HINT_SCALE, out=st.hint)
    d0, d1 = _ev(), _ev()
    torch.cuda.synchronize()
    d0.record(stream)
    for l in range(st.layers):
        draft(l, q)
    d1.record(stream)
    torch.cuda.synchronize()
    return d0.elapsed_time(d1) / st.layers


def measure_cold_start(st, tf, args, stream, world, local, steps, k0, nb, peak):
    """The same step with no cut bounds (the drafter starts every selection
    from scratch): steps/s, and the drafter per launch and back to back."""
    step_c, draft_c, kinds = make_step(st, tf, args.two_call_draft, stream, hinted=False)
    cyc = StepCycle(step_c)
    cyc.k = k0
    for _ in range(2):
        cyc()
    value, elapsed_s, _ = time_steps(cyc, steps, stream, world, local)
    per_kind = per_kernel_times(cyc, st.layers, max(3, steps // 2), kinds)
    draft = kernel_entry(nb["draft"], statistics.mean(per_kind["draft"]), peak)
    draft["back_to_back"] = kernel_entry(nb["draft"], draft_back_to_back_ms(st, draft_c, cyc, stream), peak)
    return {"value": round(value, 4), "unit": "steps/s", "steps": steps,
            "ms_per_step": round(elapsed_s / steps * 1e3, 4), "retrieval_draft": draft,
            "what": "the same step without the previous step's cut as a bound"}


def measure_extra_workload(w, args, tf, synth, dev, stream, world, local, peak):
    """The step on another workload: steps/s, the per-kernel breakdown with the
    verify roofline, and the drafter back to back."""
    import torch

    st = StepState(w, w.layers, dev, tf, synth)
    step, draft, kinds = make_step(st, tf, args.two_call_draft, stream)
    cyc = StepCycle(step)
    for _ in range(max(3, args.warmup)):
        cyc()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 2)
    value, elapsed_s, clocks = time_steps(cyc, steps, stream, world, local)
    cyc_k, kinds_k = breakdown_cycle(st, tf, args, stream, cyc.k)
    per_kind = per_kernel_times(cyc_k, st.layers, max(3, steps // 2), kinds_k)
    cyc.k = cyc_k.k
    nb = st.bytes_per_launch()
    kern = {}
    for k in kinds_k:
        name = "retrieval_draft" if k == "draft" else k
        kern[name] = kernel_entry(nb[k], statistics.mean(per_kind[k]), peak)
    kern["verify"]["calls"] = verify_label(st)
    kern["retrieval_draft"]["calls"] = draft_label(st, args.two_call_draft)
    kern["retrieval_draft"]["back_to_back"] = kernel_entry(nb["draft"], draft_back_to_back_ms(st, draft, cyc, stream),
                                                           peak)
    kern["sparse_verify_level1"] = measure_level1(st, w, tf, dev, stream, peak)
    cold = None if args.two_call_draft else measure_cold_start(st, tf, args, stream, world, local, steps, cyc.k, nb,
                                                                peak)
    ver = kern["verify"]
    out = {"value": round(value, 4), "unit": "steps/s", "steps": steps, "ms_per_step": round(elapsed_s / steps * 1e3, 4),
           "config": {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.D, "context": w.L, "layers": w.layers,
                      "ragged": bool(w.ragged), "seq_lens": st.seq_cpu.tolist(), "budget_tokens": w.budget,
                      "verify_tokens": w.T},
           "roofline": {"bound": "hbm", "kernel": verify_label(st), "achieved": ver["GBps"], "peak": peak,
                        "unit": "GB/s", "frac": ver["frac_hbm"], "algorithmic_bytes": nb["verify"],
                        "traffic": recorded_traffic("verify_attn.cu", w.name)},
           "kernels": kern, "clocks": clocks,
           "gpu_launches": steps * st.layers * launches_per_layer(st, args.two_call_draft)}
    if cold is not None:
        out["cold_start"] = cold
    kern["retrieval_draft"]["traffic"] = None if args.two_call_draft else recorded_traffic("retrieval_draft.cu",
                                                                                            w.name)
    del st
    torch.cuda.empty_cache()
    return out


def measure_offload(st, tf, stream, peak, kernels):
    """The offloaded setting on one 128K layer: the verify streamed from pinned
    host memory, the retrieval drafter's cache packed (from device memory and
    from pinned host memory), and one offloaded layer step."""
    import torch

    w, dev = st.w, st.dev
    B, Hq, Hkv, L, D, T = w.B, w.Hq, w.Hkv, w.L, w.D, w.T
    units, G = B * Hkv, Hq // Hkv
    Kh = torch.empty(st.K[0].shape, dtype=st.K.dtype, pin_memory=True)
    Vh = torch.empty(st.V[0].shape, dtype=st.V.dtype, pin_memory=True)
    Kh.copy_(st.K[0])
    Vh.copy_(st.V[0])
    off_bytes = 2 * Kh.numel() * 2
    seg_rows = min(16384, L)
    ws_off = tf.workspace(tf.tf_verify_attn_offload_workspace(B, Hq, Hkv, L, T, seg_rows), dev)
    o_off = torch.empty((B, Hq, T, D), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()
    Lmax_seq = int(st.seq_cpu.max())

    def verify_off():
        tf.tf_verify_attn_offload(st.Q[0], Kh, Vh, st.seq, Lmax_seq, st.scale, out=o_off, ws=ws_off, seg_rows=seg_rows,
                                  copy_stream=side)

    # The host link is shared with the machine's other GPUs and jobs: every
    # figure over it is the fastest of five calls (a median of three once read
    # 22 ms for a 10.3 ms call, another time the plain copy 3x slow).
    off_ms = _median_call_ms(verify_off, stream, reps=5, agg=min)
    stage = torch.empty_like(st.K[0])

    def h2d():
        stage.copy_(Kh, non_blocking=True)
        stage.copy_(Vh, non_blocking=True)

    h2d_ms = _median_call_ms(h2d, stream, reps=5, agg=min)
    del stage
    h2d_gbps = off_bytes / (h2d_ms / 1e3) / 1e9
    kernels["verify_offloaded_1layer"] = {
        "ms": round(off_ms, 4), "GBps": round(off_bytes / (off_ms / 1e3) / 1e9, 1), "h2d_copy_GBps": round(h2d_gbps, 1),
        "frac_of_h2d_copy": round(h2d_ms / off_ms, 4), "calls": "tf_verify_attn_offload",
        "timing": "K/V in pinned host memory, 16K-position segments, copies on a second stream; fastest of 5 calls "
                  "against the fastest of 5 plain pinned host-to-device copies of the same bytes"}

    # the retrieval drafter's resident cache: this layer's selection packed
    kc = w.kc
    Kc = torch.empty((B, Hkv, kc * w.chunk, D), dtype=torch.bfloat16, device=dev)
    Vc = torch.empty_like(Kc)
    lens = torch.empty(units, dtype=torch.int32, device=dev)
    nch = torch.empty(units, dtype=torch.int32, device=dev)
    nb = st.bytes_per_launch()
    rows_bytes = nb["sparse"] - B * Hkv * kc * 4 - B * Hq * D * 6  # selected K+V bytes
    pack_bytes = 2 * rows_bytes + B * Hkv * kc * 4  # read + written, ids

    def pack(src_k, src_v):
        return lambda: tf.tf_pack_retrieval_cache(src_k, src_v, st.seq, st.idx[0], st.nsel[0], Kc, Vc, lens, nch)

    pk_dev = _median_call_ms(pack(st.K[0], st.V[0]), stream)
    pk_host = _median_call_ms(pack(Kh, Vh), stream, reps=5, agg=min)
    kernels["pack_retrieval_cache_1layer"] = {
        "device": dict(kernel_entry(pack_bytes, pk_dev, peak), bytes=pack_bytes,
                       bound="selected K+V rows read and written once (HBM)"),
        "pinned_host": {"ms": round(pk_host, 5), "GBps_over_link": round(rows_bytes / (pk_host / 1e3) / 1e9, 1),
                        "frac_of_h2d_copy": round(rows_bytes / (pk_host / 1e3) / 1e9 / h2d_gbps, 4),
                        "bytes_over_link": rows_bytes,
                        "bound": "the selected rows over the host link, against a plain pinned copy"},
        "calls": "tf_pack_retrieval_cache"}

    # one offloaded layer step: refresh the drafter's packed cache from host
    # memory, the drafter over it, the tiny drafter over its resident window,
    # and the verify streamed from host memory
    win = w.n_sink + w.window
    Kw = torch.empty((B, Hkv, win, D), dtype=torch.bfloat16, device=dev)
    Vw = torch.empty_like(Kw)
    for b in range(B):
        Lb = int(st.seq_cpu[b])
        pos = list(range(0, min(w.n_sink, Lb))) + list(range(max(w.n_sink, Lb - w.window), Lb))
        Kw[b, :, : len(pos)] = st.K[0, b][:, pos]
        Vw[b, :, : len(pos)] = st.V[0, b][:, pos]
    wlens = torch.tensor([min(win, int(x)) for x in st.seq_cpu], dtype=torch.int32, device=dev)
    ident = torch.arange(kc, dtype=torch.int32, device=dev).repeat(units, 1, 1).contiguous()
    o_sp = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    o_w = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws_sp1 = tf.workspace(tf.tf_sparse_decode_attn_workspace(units, G, 1, kc), dev)
    ws_w1 = tf.workspace(tf.tf_stream_window_attn_workspace(B, Hq, Hkv, w.n_sink, w.window), dev)

    def off_step():
        tf.tf_pack_retrieval_cache(Kh, Vh, st.seq, st.idx[0], st.nsel[0], Kc, Vc, lens, nch)
        tf.tf_sparse_decode_attn(st.q[0].view(units, G, D), Kc.view(units, 1, kc * w.chunk, D),
                                 Vc.view(units, 1, kc * w.chunk, D), lens, ident, nch.view(units, 1), st.scale,
                                 out=o_sp.view(units, G, D), ws=ws_sp1)
        tf.tf_stream_window_attn(st.q[0], Kw, Vw, wlens, w.n_sink, w.window, st.scale, out=o_w, ws=ws_w1)
        verify_off()

    step_ms = _median_call_ms(off_step, stream, reps=5, agg=min)
    link = off_bytes + rows_bytes
    kernels["offloaded_step_1layer"] = {
        "ms": round(step_ms, 4), "bytes_over_link": link, "GBps_over_link": round(link / (step_ms / 1e3) / 1e9, 1),
        "frac_of_h2d_copy": round(link / (step_ms / 1e3) / 1e9 / h2d_gbps, 4),
        "calls": "tf_pack_retrieval_cache (from host) + tf_sparse_decode_attn (packed) + tf_stream_window_attn "
                 "(resident window) + tf_verify_attn_offload",
        "steps_per_s_32_layers": round(1e3 / (step_ms * w.layers), 3)}
    del Kh, Vh


def run_gpu(args):
    import torch

    sys.path.insert(0, ROOT)
    from hierarchical_speculative_decoding_gb300 import binding as tf
    from hierarchical_speculative_decoding_gb300 import synth

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    tf.load()
    w = synth.WORKLOADS[args.workload]
    layers = args.layers or w.layers
    B, Hq, Hkv, L, D, T = w.B, w.Hq, w.Hkv, w.L, w.D, w.T
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()

    st = StepState(w, layers, dev, tf, synth)
    # chunk-mean index (prefill-time; timed once for its own bandwidth)
    means_ms = _median_call_ms(lambda: tf.tf_build_chunk_means(st.K[0], st.seq, st.M[0]), stream, reps=3)
    means_bytes = B * Hkv * L * D * 2 + B * Hkv * st.Cmax * D * 2

    step, draft, kinds = make_step(st, tf, args.two_call_draft, stream)
    cyc = StepCycle(step)
    for _ in range(args.warmup):
        cyc()
    torch.cuda.synchronize()
    run_step = cyc
    graphs = []
    if args.graph:
        # the same launches, programmatic-dependent-launch edges included,
        # captured once per query set (and once on the live input buffers,
        # for the end-to-end loop); every buffer and workspace is already
        # allocated
        for k in list(range(N_QUERY_SETS)) + [None]:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(None, k)
            graphs.append(g)
        torch.cuda.synchronize()
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()

        class GraphCycle:
            def __init__(self):
                self.k = 0

            def __call__(self):
                graphs[self.k % N_QUERY_SETS].replay()
                self.k += 1

        run_step = GraphCycle()

    # ---- timed region: device-resident inputs (64 GiB of KV >> 129 MB L2)
    value, elapsed_s, clocks = time_steps(run_step, args.steps, stream, world, local)

    # ---- per-kernel breakdown and the verify roofline
    k_steps = max(3, args.steps // 2)
    cyc_k, kinds_k = breakdown_cycle(st, tf, args, stream, getattr(run_step, "k", cyc.k))
    per_kind = per_kernel_times(cyc_k, layers, k_steps, kinds_k)
    cyc.k = cyc_k.k
    nb = st.bytes_per_launch()
    kernels = {}
    for k in kinds_k:
        name = "retrieval_draft" if k == "draft" else k
        kernels[name] = kernel_entry(nb[k], statistics.mean(per_kind[k]), peak)
    kernels["retrieval_draft"]["calls"] = draft_label(st, args.two_call_draft)
    kernels["retrieval_draft"]["traffic"] = (None if args.two_call_draft
                                             else recorded_traffic("retrieval_draft.cu", w.name))
    # the two-call form of the retrieval drafter, for comparison: each call back to back over the
    # layers as one CUDA graph (eager launches with events between them timed the host's launch gaps)
    if not args.two_call_draft:
        def topk(l):
            tf.tf_chunk_scores_topk(st.q[l], st.M[l], st.seq, L, w.kc, st.idx[l], st.nsel[l], ws=st.ws_topk)

        def sparse(l):
            tf.tf_sparse_decode_attn(st.q[l], st.K[l], st.V[l], st.seq, st.idx[l], st.nsel[l], st.scale,
                                     out=st.o_sp[l], ws=st.ws_sp)

        for k, f in (("topk", topk), ("sparse", sparse)):
            ms = graph_loop_ms([lambda l=l, f=f: f(l) for l in range(layers)], stream)
            kernels["two_call_" + k] = dict(kernel_entry(nb[k], ms, peak), timing="back to back over the layers, "
                                                                                   "replayed as one CUDA graph")
    kernels["retrieval_draft"]["back_to_back"] = kernel_entry(nb["draft"], draft_back_to_back_ms(st, draft, cyc, stream),
                                                              peak)

    kernels["sparse_verify_level1"] = measure_level1(st, w, tf, dev, stream, peak)
    # the window: back to back, and its fixed cost with 4 sinks + 12 recent rows (16 rows) per unit
    ws_w16 = tf.workspace(tf.tf_stream_window_attn_workspace(B, Hq, Hkv, 4, 12), dev)
    o_w16 = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    win_ms = graph_loop_ms([lambda l=l: tf.tf_stream_window_attn(st.q[l], st.K[l], st.V[l], st.seq, w.n_sink, w.window,
                                                                 st.scale, out=st.o_win[l], ws=st.ws_win)
                            for l in range(layers)], stream)
    if "window" not in kernels:
        kernels["window"] = {"in_step": "no: the step computes the window rows inside the verify launch"}
    kernels["window"]["back_to_back"] = dict(kernel_entry(nb["window"], win_ms, peak), timing="replayed as one CUDA graph")
    kernels["window"]["floor_16rows_us"] = round(graph_loop_ms(
        [lambda l=l: tf.tf_stream_window_attn(st.q[l], st.K[l], st.V[l], st.seq, 4, 12, st.scale, out=o_w16,
                                              ws=ws_w16) for l in range(layers)], stream) * 1e3, 2)
    # the fused call against verify alone and against the two separate calls, per layer
    def ver_alone(l):
        tf.tf_verify_attn(st.Q[l], st.K[l], st.V[l], st.seq, st.scale, out=st.o_ver[l], ws=st.ws_ver)

    def separate(l):
        tf.tf_stream_window_attn(st.q[l], st.K[l], st.V[l], st.seq, w.n_sink, w.window, st.scale, out=st.o_win[l],
                                 ws=st.ws_win)
        ver_alone(l)

    def fused(l):
        tf.tf_verify_window_attn(st.Q[l], st.q[l], st.K[l], st.V[l], st.seq, w.n_sink, w.window, st.scale,
                                 out=st.o_ver[l], wout=st.o_win[l], ws=st.ws_vw)

    kernels["verify"]["back_to_back_us"] = {
        name: round(graph_loop_ms([lambda l=l, f=f: f(l) for l in range(layers)], stream) * 1e3, 2)
        for name, f in (("verify_window_one_call", fused), ("verify_alone", ver_alone),
                        ("window_then_verify", separate))}
    kernels["verify"]["calls"] = verify_label(st)

    # the offloaded setting (one 128K layer; not part of the step)
    measure_offload(st, tf, stream, peak, kernels)
    kernels["chunk_means_prefill_1layer"] = {"ms": round(means_ms, 4),
                                             "GBps": round(means_bytes / (means_ms / 1e3) / 1e9, 1)}
    ver_ms = statistics.mean(per_kind["verify"])
    achieved = nb["verify"] / (ver_ms / 1e3) / 1e9
    traffic = recorded_traffic("verify_attn.cu", w.name)

    result = {
        "metric": METRIC, "value": round(value, 4), "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_s / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "Hq": Hq, "Hkv": Hkv, "head_dim": D, "context": L, "layers": layers,
                   "chunk": w.chunk, "budget_tokens": w.budget, "window": f"{w.n_sink}+{w.window}",
                   "verify_tokens": T, "l2": "inputs larger than L2: 2 GiB of K+V per layer, no flush needed",
                   "launch": "one CUDA graph per step" if args.graph else "stream launches",
                   "queries": f"{N_QUERY_SETS} seeded query sets cycled over the steps; the retrieval drafter "
                              f"takes the previous step's cut x {HINT_SCALE} of each layer as a bound "
                              f"(cold_start: the same step without it)"},
        "roofline": {"bound": "hbm", "kernel": verify_label(st), "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": nb["verify"], "peak_source": peak_kind},
        "kernels": kernels,
        "kernel_timing": f"CUDA events around every launch, {k_steps} further steps after the timed region",
        "gpu_launches": args.steps * layers * launches_per_layer(st, args.two_call_draft),
        "clocks": clocks,
    }

    # ---- accept / resample (latency-bound; reported in microseconds per call):
    # the two-level step of a batch of 8 over vocabulary 32000, gamma 4 then 5,
    # and the tree form on a binary tree of 14 candidates
    acc = synth.two_level_inputs(8, 4, w.vocab, seed=4, device=dev)
    q_lvl1 = acc["q"][:, :5].contiguous()
    ws_a1 = tf.workspace(tf.tf_spec_accept_workspace(8, 4), dev)
    ws_a2 = tf.workspace(tf.tf_spec_accept_workspace(8, 5), dev)
    outs1 = [torch.empty(8, dtype=torch.int32, device=dev) for _ in range(2)] + [
        torch.empty((8, 5), dtype=torch.int32, device=dev)]
    outs2 = [torch.empty(8, dtype=torch.int32, device=dev) for _ in range(2)] + [
        torch.empty((8, 6), dtype=torch.int32, device=dev)]

    def two_level():
        tf.tf_spec_accept(q_lvl1, acc["r"], acc["x"], acc["u1"], acc["ur1"], n_acc=outs1[0], next_token=outs1[1],
                          out_tokens=outs1[2], ws=ws_a1)
        tf.tf_spec_accept(acc["p"], acc["q"], outs1[2], acc["u2"], acc["ur2"], n_acc=outs2[0], next_token=outs2[1],
                          out_tokens=outs2[2], ws=ws_a2)

    def per_call_us(fn, n=20):
        return round(graph_loop_ms([fn] * n, stream) * 1e3, 2)

    kernels["spec_accept_two_level_b8_v32000"] = {"us_per_step": per_call_us(two_level), "launches_per_step": 4,
                                                  "timing": "20 steps replayed as one CUDA graph"}
    tri = synth.tree_accept_inputs(8, 14, w.vocab, seed=5, device=dev, branching=2)
    ws_t = tf.workspace(tf.tf_spec_accept_tree_workspace(8, 14, w.vocab), dev)
    t_out = [torch.empty(8, dtype=torch.int32, device=dev) for _ in range(2)] + [
        torch.empty((8, 15), dtype=torch.int32, device=dev), torch.empty((8, 14), dtype=torch.int32, device=dev)]

    def tree_accept():
        tf.tf_spec_accept_tree(tri["tgt"], tri["drf"], tri["x"], tri["parent"], tri["u_acc"], tri["u_res"],
                               n_acc=t_out[0], next_token=t_out[1], out_tokens=t_out[2], acc_nodes=t_out[3], ws=ws_t)

    kernels["spec_accept_tree_binary_t14_b8_v32000"] = {"us_per_call": per_call_us(tree_accept),
                                                         "launches_per_call": 2,
                                                         "timing": "20 calls replayed as one CUDA graph"}

    # ---- end to end through the public API with host buffers: every step
    # copies its query set from pinned host memory into the live buffers
    if not args.no_e2e:
        q_host = st.q_sets.cpu().pin_memory()
        Q_host = st.Q_sets.cpu().pin_memory()
        outs_host = [t.cpu().pin_memory() for t in (st.o_sp, st.o_win, st.o_ver)]
        h2d = q_host[0].numel() * 2 + Q_host[0].numel() * 2
        d2h = sum(t.numel() * 4 for t in outs_host)
        e_steps = max(3, args.steps // 2)
        # the step with its copies as one CUDA graph per query set (every call takes caller-owned
        # buffers and workspaces, so the step captures as is); one launch and one host wait per step
        e_graphs = e2e_graphs(st, step, q_host, Q_host, outs_host)
        for g in e_graphs:
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(e_steps):
            e_graphs[i % N_QUERY_SETS].replay()
            torch.cuda.current_stream().synchronize()
        e_value, _ = job_throughput(e_steps, time.perf_counter() - t0, world)
        result["e2e"] = {"value": round(e_value, 4), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h,
                         "what": "per step, one CUDA graph: the queries copied from pinned host memory, each "
                                 "layer's outputs copied back on a copy stream after the layer (overlapping the next "
                                 "layers), then a host wait for the last copy"}

    if not args.two_call_draft:
        result["cold_start"] = measure_cold_start(st, tf, args, stream, world, local, k_steps, cyc.k + 1, nb, peak)
    del st, run_step, step, draft, cyc, graphs
    torch.cuda.empty_cache()

    # ---- the other workloads, one after the other (each frees its cache)
    extra = [x for x in args.extra_workloads.split(",") if x and x != "none" and x != w.name]
    if extra and args.layers is None:
        result["workloads"] = {}
        for name in extra:
            result["workloads"][name] = measure_extra_workload(synth.WORKLOADS[name], args, tf, synth, dev, stream,
                                                               world, local, peak)

    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm


def run_reference(args):
    """The float64 oracle on every host core; each step is one batch of
    (layer, KV head) units (one per worker), scaled to a full step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    sys.path.insert(0, ROOT)
    from hierarchical_speculative_decoding_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    # the oracle has no warm state; the pool's workers import everything before
    # the clock starts
    cb = cpu_baseline(w, units_per_worker=max(1, args.steps))
    step_s = 1.0 / cb["value"]
    out = {"metric": METRIC, "value": cb["value"], "unit": "steps/s", "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.D, "context": w.L,
                      "layers": w.layers, "chunk": w.chunk, "budget_tokens": w.budget,
                      "window": f"{w.n_sink}+{w.window}", "verify_tokens": w.T},
           "cpu_baseline": cb,
           "e2e": {"value": cb["value"], "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_gpu(a)
