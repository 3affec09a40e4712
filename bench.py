"""Benchmark of the emulated Ulysses attention hot path on GB300.

One step = the whole path of one attention layer, forward and backward, over
one batch of seeded synthetic input already resident in HBM:
  q/k/v exchange (seq -> head) · document boundaries from the gathered
  position_ids · attention forward · O exchange (head -> seq) · dO exchange
  (seq -> head) · attention backward (D rows, dK/dV, dQ, dsinks) · dQ/dK/dV
  exchanges (head -> seq).

The headline value is the attention's algorithmic fwd+bwd work,
14 * D * Hq * (visible query/key pairs), divided by the whole step's time,
in TFLOP/s.  The same JSON line carries the relayout bandwidth, per-call
times, the roofline of the dominant kernel, an end-to-end figure measured
through the C ABI with host buffers, and the fp64 oracle's CPU throughput.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       python bench.py --impl reference ...   (the oracle on the host cores)
For N > 1 each rank runs its own replica of the emulated P-rank job on its
own GPU (no collective on the data path; barrier + max-over-ranks timing).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import usp_workloads as W  # noqa: E402

DEFAULT_WORKLOAD = W.LLAMA32K.name
METRIC = "varlen GQA attention fwd+bwd TFLOP/s at 1 GB300; relayout GB/s"


# ----------------------------------------------------------------------------- host-side counts
def visible_pairs(w: W.Workload) -> int:
    """Query/key pairs the mask keeps, from the seeded document lengths (closed forms)."""
    total = 0
    for lens in W.document_lengths(w):
        for L in lens:
            if w.window_left < 0:
                total += L * (L + 1) // 2 if w.causal else L * L
            else:
                wl = w.window_left
                if w.causal:
                    m = min(L, wl + 1)               # rows i < wl+1 see i+1 keys, the rest wl+1
                    total += m * (m + 1) // 2 + (L - m) * (wl + 1)
                else:
                    total += sum(min(L - 1, i + wl) - max(0, i - wl) + 1 for i in range(L))
    return total


def attention_flops(w: W.Workload):
    pairs = visible_pairs(w)
    unit = w.D * w.Hq * pairs
    # forward QK^T + PV = 4 flops per pair and dim; backward recompute S, dP, dV,
    # dK, dQ = 10; of the backward, the dK/dV kernel does S, dP, dV, dK (8) and
    # the dQ kernel does the one remaining algorithmic GEMM, dQ (2).
    return {"pairs": pairs, "fwd": 4 * unit, "bwd": 10 * unit, "total": 14 * unit,
            "dkdv": 8 * unit, "dq": 2 * unit}


def relayout_bytes(w: W.Workload):
    q = w.B * w.S * w.Hq * w.D * 2
    kv = w.B * w.S * w.Hkv * w.D * 2
    rep = max(1, w.P // w.Hkv)  # key/value heads replicated when there are fewer than ranks
    # every exchange reads and writes each element once; a replicated head is
    # written (forward) or read (backward) once per replica
    return {"qkv": 2 * q + 2 * (kv + rep * kv), "o": 2 * q, "do": 2 * q, "dqkv": 2 * q + 2 * (rep * kv + kv)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- the step
CALLS = ["relayout_qkv", "cu_seqlens", "attn_fwd", "relayout_o", "relayout_do", "attn_bwd_pre", "attn_bwd_dkdv",
         "attn_bwd_dq", "relayout_dqkv"]


L2_BYTES = 129 * 1024 * 1024


def relayout_bandwidth(w: W.Workload, device, t, steps: int):
    """GB/s of the explicit exchange kernels alone: the q/k/v exchange
    (seq -> head) and the O exchange (head -> seq), `steps` times each after
    three warm-up rounds.  Every element is read once and written once.

    When the tensors the exchanges touch fit in twice the L2 (the 4K MHA
    workload's 12.6 MB tensors), L2 is flushed before every round (a 256 MB
    buffer is written) and each round is timed on its own with CUDA events;
    otherwise the rounds run back to back.  Returns (GB/s, ms per round, how
    L2 was handled)."""
    from ulysses_sequence_long_gb300.pipeline import Shape, UlyssesAttention
    ua = UlyssesAttention(Shape(w.B, w.S, w.Hq, w.Hkv, w.D, w.P, w.causal, w.window_left), device=device,
                          with_backward=False, fused=False)
    s = torch.cuda.current_stream(device)
    ua.o_head.zero_()
    rb = relayout_bytes(w)
    touched = (rb["qkv"] + rb["o"])
    flush = touched < 2 * L2_BYTES
    scrub = torch.empty((256 * 1024 * 1024,), dtype=torch.uint8, device=device) if flush else None
    for _ in range(3):
        ua.exchange_qkv(t["q"], t["k"], t["v"], s)
        ua.exchange_out(s)
    torch.cuda.synchronize()
    if flush:
        times = []
        for _ in range(steps):
            scrub.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            ua.exchange_qkv(t["q"], t["k"], t["v"], s)
            ua.exchange_out(s)
            b.record(s)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        how = "L2 flushed (256 MB written) before every round, median of per-round CUDA events"
    else:
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s)
        for _ in range(steps):
            ua.exchange_qkv(t["q"], t["k"], t["v"], s)
            ua.exchange_out(s)
        stop.record(s)
        torch.cuda.synchronize()
        ms = start.elapsed_time(stop) / steps
        how = "tensors larger than L2, rounds back to back"
    del ua, scrub
    torch.cuda.empty_cache()
    return touched / (ms * 1e-3) / 1e9, ms, how


def scan_positions(n: int, mean: int = 4096, seed: int = 11, device="cuda"):
    """position_ids of n tokens packed with documents of geometric lengths
    (mean `mean`, seeded), built on the device: positions count from 0 in
    each document.  Returns (positions int32 [n], number of documents)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens, tot = [], 0
    while tot < n:
        L = min(int(rng.geometric(1.0 / mean)), n - tot)
        lens.append(L)
        tot += L
    lens_t = torch.tensor(lens, dtype=torch.int64, device=device)
    starts = torch.cumsum(lens_t, 0) - lens_t
    pos = torch.arange(n, dtype=torch.int64, device=device) - torch.repeat_interleave(starts, lens_t)
    return pos.to(torch.int32), len(lens)


def scan_bandwidth(device, reps: int = 10, n: int = 1 << 28):
    """GB/s of the document-boundary scan alone over n positions (1 GiB at
    2^28), L2 flushed before every call: 4n bytes read plus 4(docs+1)
    written per call, median of per-call CUDA events."""
    from ulysses_sequence_long_gb300 import binding as B
    pos, docs = scan_positions(n, device=device)
    cu = torch.empty((n + 1,), dtype=torch.int32, device=device)
    nd = torch.zeros(1, dtype=torch.int32, device=device)
    mx, st = torch.zeros_like(nd), torch.zeros_like(nd)
    ws = torch.empty((B.usp_cu_seqlens_workspace_bytes(1, n),), dtype=torch.uint8, device=device)
    scrub = torch.empty((256 * 1024 * 1024,), dtype=torch.uint8, device=device)
    times = []
    for r in range(reps + 3):
        scrub.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        B.usp_cu_seqlens_from_position_ids(pos, 1, n, 8, cu, nd, mx, ws, st)
        b.record()
        torch.cuda.synchronize()
        if r >= 3:
            times.append(a.elapsed_time(b))
    assert int(st.item()) == 0 and int(nd.item()) == docs, "scan sweep: wrong document count"
    ms = statistics.median(times)
    byts = 4 * n + 4 * (docs + 1)
    del pos, cu, ws, scrub
    torch.cuda.empty_cache()
    return {"tokens": n, "documents": docs, "ms": ms, "gbs": byts / (ms * 1e-3) / 1e9,
            "how": "one call over 2^28 positions, L2 flushed before each, median of CUDA events"}


class Step:
    def __init__(self, w: W.Workload, device, host=None, fused=None):
        from ulysses_sequence_long_gb300.pipeline import HybridAttention, Shape, UlyssesAttention
        self.w = w
        self.device = device
        shape = Shape(w.B, w.S, w.Hq, w.Hkv, w.D, w.P, w.causal, w.window_left)
        self.hybrid = w.ring > 1
        if self.hybrid:   # ring x Ulysses: the Ulysses exchange inside each ring group
            self.ua = HybridAttention(shape, w.ring, device=device, fused=fused)
        else:
            self.ua = UlyssesAttention(shape, device=device, fused=fused)
        if host is None:
            host = {"t": W.qkv_do_shards(w), "pos": torch.from_numpy(W.position_ids_shards(w)), "sinks": W.sinks(w)}
        self.shared_host = host
        self.host = host["t"]
        self.dev = {n: x.to(device) for n, x in self.host.items()}
        self.pos_host = host["pos"]
        self.pos = self.pos_host.to(device)
        sk = host["sinks"]
        self.sinks = None if sk is None else sk.to(device)
        self.stream = torch.cuda.current_stream(device)
        self.n_events = 0

    def run(self, events=None, group_events=None):
        """One whole step; optional CUDA events recorded between the calls
        (event i+1 closes CALLS[i]; exchanges that the fused mode folds into
        the attention kernels take ~0 ms).  When the backward runs in
        key/value head groups, group_events[g][0] / [1] close group g's dK/dV
        and dQ passes."""
        ua, d, s = self.ua, self.dev, self.stream

        def mark(i):
            if events is not None:
                events[i].record(s)

        def gmark(g, i):
            if group_events is not None:
                group_events[g][i].record(s)

        if self.hybrid:
            ua.forward_phases(d["q"], d["k"], d["v"], self.pos, self.sinks, s, marks=mark)
            ua.backward_phases(d["do"], self.sinks, s, marks=lambda i: mark(4 + i))
            return
        mark(0)
        ua.exchange_qkv(d["q"], d["k"], d["v"], s)
        mark(1)
        ua.boundaries(self.pos, s)
        mark(2)
        ua.attention(self.sinks, s)
        mark(3)
        ua.exchange_out(s)
        ua.backward_phases(d["do"], self.sinks, s, marks=lambda i: mark(4 + i), group_marks=gmark)

    def launches_per_step(self) -> int:
        sink = 1 if self.sinks is not None else 0
        extra = 2 * (len(self.ua.ds_groups) - 1)   # dK/dV + dQ of each further key/value head group
        # the scan is one launch up to 32768 positions (one block), else a
        # state reset and the scan
        scan = 1 if self.w.B * self.w.S <= 32768 else 2
        if self.hybrid:
            # scan, preprocess 1 (+ dsink); per ring step: forward + merge,
            # dK/dV + 2 sums, dQ + 1 sum; explicit exchanges add 1 + 1 + 1 + 3
            return scan + 1 + sink + (7 + extra) * self.w.ring + (2 if self.ua.fused else 6)
        # scan, fwd 1, preprocess 1 (+ dsink 1), dK/dV 1, dQ 1; the fused
        # step adds the k/v exchange for the forward (2), the explicit one
        # relayout qkv 1, O 1, dO 1, dQ/dK/dV 3
        return scan + 4 + sink + extra + (2 if self.ua.fused else 6)

    # -- end to end: host buffers in and out, through the C ABI
    def make_host_io(self):
        pin = {n: x.pin_memory() for n, x in self.host.items()}
        pin["pos"] = self.pos_host.pin_memory()
        ua = self.ua
        outs = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for n, t in (("o", ua.o_seq), ("dq", ua.dq_seq), ("dk", ua.dk_seq), ("dv", ua.dv_seq))}
        if self.sinks is not None:
            outs["dsinks"] = torch.empty(ua.dsinks.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        return pin, outs, h2d, d2h

    def upload(self, pin):
        d = self.dev
        for n in ("q", "k", "v", "do"):
            d[n].copy_(pin[n], non_blocking=True)
        self.pos.copy_(pin["pos"], non_blocking=True)

    def download(self, outs):
        ua = self.ua
        outs["o"].copy_(ua.o_seq, non_blocking=True)
        outs["dq"].copy_(ua.dq_seq, non_blocking=True)
        outs["dk"].copy_(ua.dk_seq, non_blocking=True)
        outs["dv"].copy_(ua.dv_seq, non_blocking=True)
        if "dsinks" in outs:
            outs["dsinks"].copy_(ua.dsinks, non_blocking=True)


def run_e2e(slots, pin, outs, steps):
    """`steps` whole steps with host buffers in and out, double-buffered.

    Every step uploads its inputs from pinned host memory and downloads its
    results (O, dQ, dK, dV, dsinks) to pinned host memory.  Step k computes on
    slot k%2 while the inputs of step k+1 upload on one copy stream and the
    results of step k-1 download on another.  Returns the elapsed ms between
    CUDA events recorded before the first upload and after the last download.
    """
    comp = slots[0].stream
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(comp)
    up.wait_event(start)
    with torch.cuda.stream(up):
        slots[0].upload(pin)
        in_ready[0].record(up)
    for k in range(steps):
        c, n = k % 2, (k + 1) % 2
        comp.wait_event(in_ready[c])
        if k >= 2:
            comp.wait_event(out_read[c])         # results of step k-2 have left this slot
        with torch.cuda.stream(comp):
            slots[c].run()
        done[c].record(comp)
        if k + 1 < steps:
            if k >= 1:
                up.wait_event(done[n])           # step k-1 no longer reads that slot's inputs
            with torch.cuda.stream(up):
                slots[n].upload(pin)
                in_ready[n].record(up)
        down.wait_event(done[c])
        with torch.cuda.stream(down):
            slots[c].download(outs)
            out_read[c].record(down)
    comp.wait_stream(down)
    stop.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(stop)


def run_e2e_serial(step, pin, outs, steps):
    """Per-step latency with host buffers: upload, the whole step and the
    download run one after another on one stream, nothing overlapped.
    Returns the mean ms of one such step (CUDA events around each)."""
    s = step.stream
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        with torch.cuda.stream(s):
            step.upload(pin)
            step.run()
            step.download(outs)
        b.record(s)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.mean(times)


# ----------------------------------------------------------------------------- oracle timing
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def _oracle_threads() -> int:
    """Threads the oracle's numpy BLAS pool runs with: threadpoolctl's report
    when it is installed, else the thread-count variable this process was
    started with, else every host core (the BLAS default)."""
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        for v in _THREAD_VARS:
            if os.environ.get(v, "").isdigit():
                return int(os.environ[v])
        return os.cpu_count() or 1


def oracle_sample(w: W.Workload, budget_s: float = 20.0):
    """Time the fp64 oracle (as it stands) on a bounded sample of the workload.

    The sample is the first document of the first key/value group of rank 0
    (all of its query heads), forward and backward, grown from 512 tokens
    (doubling, at most the document) until one run takes a quarter of
    budget_s.  Returns the throughput in the bench's unit (algorithmic TFLOP/s
    of the sample) and the threads the oracle's BLAS used.
    """
    import oracle
    lens = W.document_lengths(w)[0]
    L = lens[0]
    G = w.Hq // w.Hkv
    rng = np.random.Generator(np.random.PCG64(5))
    n = min(L, 512)
    while True:
        q = rng.standard_normal((n, G, w.D))
        k = rng.standard_normal((n, 1, w.D))
        v = rng.standard_normal((n, 1, w.D))
        do = rng.standard_normal((n, G, w.D))
        t0 = time.perf_counter()
        O, Lse = oracle.attention_fwd(q, k, v, [0, n], w.causal, w.window_left)
        oracle.attention_bwd(q, k, v, O, Lse, do, [0, n], w.causal, w.window_left)
        dt = time.perf_counter() - t0
        ww = W.Workload("sample", B=1, S=n, Hq=G, Hkv=1, D=w.D, P=1, causal=w.causal, window_left=w.window_left)
        flops = attention_flops(ww)["total"]
        if dt > budget_s / 4 or n >= L:
            break
        n = min(L, n * 2)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": f"first document of rank 0, kv group 0 ({G} query heads, D={w.D}), first {n} tokens, "
                      f"fp64 numpy forward+backward, {dt:.2f} s"}


def oracle_bandwidth_parts(w: W.Workload):
    """The oracle's exchange and document-boundary scan on the whole workload:
    relayout_fwd of q, k, v plus relayout_bwd of an O-shaped tensor (the same
    bytes the GPU relayout figure counts), and cu_seqlens_from_position_ids
    over every position.  The exchanges are permutations, so they run on the
    bf16 bit patterns (uint16)."""
    import oracle
    t = W.qkv_do_shards(w, names=("q", "k", "v"))
    x = {n: t[n].view(torch.int16).numpy() for n in t}
    rep = w.Hkv < w.P
    t0 = time.perf_counter()
    qh = oracle.relayout_fwd(x["q"], w.P)
    oracle.relayout_fwd(x["k"], w.P, replicate=rep)
    oracle.relayout_fwd(x["v"], w.P, replicate=rep)
    oracle.relayout_bwd(qh, w.P)
    dt_relayout = time.perf_counter() - t0
    rb = relayout_bytes(w)
    pos = W.position_ids_shards(w)
    t0 = time.perf_counter()
    oracle.cu_seqlens_from_position_ids(pos)
    dt_scan = time.perf_counter() - t0
    return {"relayout": {"gbs": (rb["qkv"] + rb["o"]) / dt_relayout / 1e9, "seconds": dt_relayout,
                         "bytes": rb["qkv"] + rb["o"], "what": "q/k/v exchange + O exchange, whole workload"},
            "cu_seqlens": {"seconds": dt_scan, "tokens": w.B * w.S,
                           "what": "sequential scan over every gathered position"}}


def _oracle_sample_in_child(w: W.Workload, budget_s: float, threads: int):
    """oracle_sample in a fresh interpreter whose BLAS pool is fixed to
    `threads` threads by the environment (read when numpy loads its BLAS)."""
    env = dict(os.environ)
    for v in _THREAD_VARS:
        env[v] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", w.name,
                        "--oracle-budget", str(budget_s)], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(w: W.Workload, budget_s: float = 20.0):
    """The oracle as it stands, on this host's cores: the attention sample
    with a BLAS thread per host core and with one thread (each in a fresh
    interpreter with the thread count fixed), plus the whole-workload exchange
    and scan times (these are single-threaded numpy copies and a Python loop)."""
    cores = os.cpu_count() or 1
    line = _oracle_sample_in_child(w, budget_s, cores)
    line["host_cores"] = cores
    one = _oracle_sample_in_child(w, budget_s / 4, 1)
    line["single_thread"] = {"value": one["value"], "cores": one["cores"], "sample": one["sample"]}
    line.update(oracle_bandwidth_parts(w))
    return line


def rank_sync(world: int, device):
    """barrier() and max_over_ranks(x) over the job's ranks (no-ops for one
    rank): every rank runs the whole emulated layer, the job's time is the
    slowest rank's."""
    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        if world == 1:
            return x
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_over_ranks


def job_tflops(flop_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own copy of the step."""
    return flop_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per = []
    # every step is a bounded sample; the whole run stays within about two minutes
    budget = max(1.0, min(8.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, budget_s=budget)
    for _ in range(args.steps):
        per.append(oracle_sample(w, budget_s=budget))
    val = statistics.median(p["value"] for p in per)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
            "data": "synthetic (seeded N(0,1))", "scaling": "weak",
            "config": {"workload": w.name, **w.describe()},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": per[-1]["cores"], "kind": "oracle",
                             "sample": per[-1]["sample"], "host_cores": os.cpu_count() or 1},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- one workload
def attention_bytes(w: W.Workload) -> int:
    """Algorithmic HBM bytes of one fwd+bwd: the forward reads q, k, v and
    writes O and LSE; the backward reads q, k, v, O, dO and LSE and writes dQ,
    dK, dV and the D statistic (each tensor once)."""
    q = w.B * w.S * w.Hq * w.D * 2
    kv = w.B * w.S * w.Hkv * w.D * 2
    stat = w.B * w.S * w.Hq * 4
    return (2 * q + 2 * kv + stat) + (3 * q + 2 * kv + stat) + (q + 2 * kv + stat)


def measure(w: W.Workload, device, steps: int, warmup: int, fused, world: int, barrier, max_over_ranks,
            clock_index: int = 0):
    """Time `steps` whole steps of workload `w` after `warmup` untimed ones.

    Returns the Step (still holding its buffers) and the figures of the
    workload: ms per step (max over ranks), per-call ms, TFLOP/s of the step
    and of its forward and backward, and the dominant attention kernel with
    its achieved TFLOP/s against the measured burst and sustained bf16 peaks
    and against min(tensor peak, arithmetic intensity x HBM copy bandwidth).
    """
    step = Step(w, device, fused=fused)
    fl = attention_flops(w)
    for _ in range(max(warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    assert step.ua.read_status() == 0, "device status set during warm-up"
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(steps)]
    n_groups = len(step.ua.ds_groups)
    gev = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_groups)]
           for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(clock_index) as clocks:   # clocks sampled during the timed steps only
        barrier()
        torch.cuda.synchronize()
        start.record()
        for k in range(steps):
            step.run(ev[k], gev[k] if n_groups > 1 else None)
        stop.record()
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(start.elapsed_time(stop) / steps)
    assert step.ua.read_status() == 0, "device status set during the timed steps"
    per_call = {}
    for i, name in enumerate(CALLS):
        per_call[name] = statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(steps))
    if n_groups > 1 and not step.hybrid:   # the passes alternate group by group
        dkdv_i = CALLS.index("attn_bwd_dkdv")
        t_dkdv, t_dq = [], []
        for k in range(steps):
            prev, a, b = ev[k][dkdv_i], 0.0, 0.0
            for g in range(n_groups):
                a += prev.elapsed_time(gev[k][g][0])
                b += gev[k][g][0].elapsed_time(gev[k][g][1])
                prev = gev[k][g][1]
            t_dkdv.append(a)
            t_dq.append(b)
        per_call["attn_bwd_dkdv"], per_call["attn_bwd_dq"] = statistics.mean(t_dkdv), statistics.mean(t_dq)

    peaks = measured_peaks()
    attn_ms = per_call["attn_fwd"] + per_call["attn_bwd_pre"] + per_call["attn_bwd_dkdv"] + per_call["attn_bwd_dq"]
    bwd_ms = per_call["attn_bwd_pre"] + per_call["attn_bwd_dkdv"] + per_call["attn_bwd_dq"]
    kernels = {"attn_fwd": fl["fwd"], "attn_bwd_dkdv": fl["dkdv"], "attn_bwd_dq": fl["dq"]}
    dom = max(kernels, key=lambda n: per_call[n])
    achieved = kernels[dom] / (per_call[dom] * 1e-3) / 1e12
    ai = fl["total"] / attention_bytes(w)
    attainable = min(peaks["bf16_tflops"], ai * peaks["hbm_gbs"] / 1e3)
    r = {"workload": w.name, "steps": steps, "warmup": max(warmup, 3), "ms_per_step": ms,
         "tflops": job_tflops(fl["total"], world, ms), "fwd_bwd_flop": fl["total"],
         "visible_pairs_per_head": fl["pairs"],
         "fwd_tflops": fl["fwd"] / (per_call["attn_fwd"] * 1e-3) / 1e12,
         "bwd_tflops": fl["bwd"] / (bwd_ms * 1e-3) / 1e12,
         "attention_tflops": fl["total"] / (attn_ms * 1e-3) / 1e12,
         "per_call_ms": per_call,
         "dominant": {"kernel": dom, "achieved_tflops": achieved,
                      "frac_burst": achieved / peaks["bf16_tflops"],
                      "frac_sustained": achieved / peaks["bf16_tflops_sustained"]},
         "step_frac_burst": job_tflops(fl["total"], 1, ms) / peaks["bf16_tflops"],
         "arithmetic_intensity_flop_per_byte": ai,
         "attainable_tflops": attainable,
         "step_frac_attainable": job_tflops(fl["total"], 1, ms) / attainable,
         "exchanges": "fused" if step.ua.fused else "explicit",
         "dq_pass": ("recomputed S and dP" if not step.ua.stored_ds else
                     "stored dS" if n_groups == 1 else f"stored dS, {n_groups} key/value head groups"),
         "launches_per_step": step.launches_per_step(), "clocks": clocks.summary()}
    return step, r


PER_CONFIG_STEPS = {W.TINY.name: 20, W.MHA4K.name: 20, W.GPTOSS_WIN.name: 20, W.GPTOSS_FULL.name: 10,
                    W.LLAMA32K.name: 10, W.LONG128K.name: 3}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="usp", choices=["usp", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--bandwidth", default=None, choices=["relayout", "scan"],
                    help="time only the explicit exchange of --workload (L2 flushed) or the scan over 2^28 positions")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' figures (per_config)")
    ap.add_argument("--oracle-sample", default=None, help=argparse.SUPPRESS)   # internal: one oracle sample
    ap.add_argument("--oracle-budget", type=float, default=20.0, help=argparse.SUPPRESS)
    ap.add_argument("--exchange", default="auto", choices=["auto", "fused", "explicit"],
                    help="fused: attention kernels read/write the sequence shards; explicit: relayout kernels")
    args = ap.parse_args()
    if args.oracle_sample is not None:
        print(json.dumps(oracle_sample(W.BY_NAME[args.oracle_sample], args.oracle_budget)))
        return 0
    w = W.BY_NAME[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    barrier, max_over_ranks = rank_sync(world, device)

    from ulysses_sequence_long_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier()
    _build.build()

    fused = {"auto": None, "fused": True, "explicit": False}[args.exchange]
    peaks = measured_peaks()
    rb = relayout_bytes(w)
    if args.bandwidth is not None:   # one bandwidth kernel alone (for profiler captures)
        if args.bandwidth == "scan":
            r = scan_bandwidth(device, args.steps)
        else:
            t = {n: x.to(device) for n, x in W.qkv_do_shards(w, names=("q", "k", "v")).items()}
            g, ms, how = relayout_bandwidth(w, device, t, args.steps)
            r = {"workload": w.name, "ms": ms, "gbs": g, "how": how}
        r["frac_hbm"] = r["gbs"] / peaks["hbm_gbs"]
        if rank == 0:
            print(json.dumps({"bandwidth": args.bandwidth, **r}))
        return 0

    # ---- timed region of the headline workload: K whole steps, events between the calls
    step, m = measure(w, device, args.steps, args.warmup, fused, world, barrier, max_over_ranks, local)
    ms, per_call, fl = m["ms_per_step"], m["per_call_ms"], attention_flops(w)

    if step.ua.fused:
        relayout_gbs, relayout_ms, relayout_l2 = relayout_bandwidth(w, device, step.dev, args.steps)
        relayout_note = "explicit q/k/v + O exchanges timed apart (the step folds them into the attention I/O)"
    else:
        relayout_ms = (per_call["relayout_qkv"] + per_call["relayout_o"] + per_call["relayout_do"] +
                       per_call["relayout_dqkv"])
        relayout_gbs = (rb["qkv"] + rb["o"] + rb["do"] + rb["dqkv"]) / (relayout_ms * 1e-3) / 1e9
        relayout_note, relayout_l2 = "the step's six exchange launches", "inputs larger than L2"
    dom = m["dominant"]["kernel"]
    achieved = m["dominant"]["achieved_tflops"]
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tr = json.load(f)
        ent = tr.get(w.name, {}).get(dom)
        if ent is not None and ent.get("source_hash") == _build.source_hash():
            traffic = ent["bytes_per_launch"]
    # The timed region is well under a second at full clock, so the headline
    # fraction is against the burst peak; the sustained one is given beside it.
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": peaks["source"] + " bf16 burst (headline)",
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                "peak_sustained_source": peaks["source"] + " bf16 sustained"}

    line = {"metric": METRIC, "value": m["tflops"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), position_ids resets)",
            "config": {"workload": w.name, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "P": w.P,
                       "causal": w.causal, "window_left": w.window_left, "sinks": w.sinks,
                       "documents": len(W.document_lengths(w)[0]), "visible_pairs_per_head": fl["pairs"],
                       "fwd_bwd_flop": fl["total"], "parallelism": f"emulated ulysses P={w.P}, replicas={world}",
                       "exchanges": m["exchanges"], "ring": w.ring, "dq_pass": m["dq_pass"],
                       "l2": "inputs larger than L2 (no flush)"},
            "relayout_gbs": relayout_gbs, "relayout_frac_hbm": relayout_gbs / peaks["hbm_gbs"],
            "relayout_measured": relayout_note, "relayout_l2": relayout_l2,
            "attention_tflops": m["attention_tflops"], "fwd_tflops": m["fwd_tflops"], "bwd_tflops": m["bwd_tflops"],
            "per_call_ms": per_call, "roofline": roofline,
            "gpu_launches": step.launches_per_step() * args.steps, "clocks": m["clocks"]}

    if not args.no_e2e:
        pin, outs, h2d, d2h = step.make_host_io()
        twin = Step(w, device, host=step.shared_host, fused=fused)
        slots = [step, twin]
        run_e2e(slots, pin, outs, 3)               # warm-up of the copy path
        barrier()
        torch.cuda.synchronize()
        ems = run_e2e(slots, pin, outs, args.steps) / args.steps
        barrier()
        ems = max_over_ranks(ems)
        lat = max_over_ranks(run_e2e_serial(step, pin, outs, max(3, min(args.steps, 10))))
        line["e2e"] = {"value": job_tflops(fl["total"], world, ems), "unit": "TFLOP/s", "ms_per_step": ems,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "overlapped": True,
                       "how": "two buffer slots: step k computes while step k+1 uploads and step k-1 downloads "
                              "(pinned host memory, copy streams); value = steps / elapsed",
                       "latency_ms": lat, "latency_value": job_tflops(fl["total"], world, lat),
                       "latency_how": "one step with its upload and download serialised on one stream"}
        del twin, slots, pin, outs
    del step
    torch.cuda.empty_cache()

    # ---- every other workload, a few steps each (replicas time the same way)
    if not args.no_per_config:
        per = {}
        for ow in W.ALL:
            if ow.name == w.name:
                continue
            ost, om = measure(ow, device, PER_CONFIG_STEPS.get(ow.name, 5), args.warmup, fused, world,
                              barrier, max_over_ranks, local)
            if ost.ua.fused:
                g, _, how = relayout_bandwidth(ow, device, ost.dev, 10)
            else:
                g, how = None, "explicit exchanges inside the step: see per_call_ms"
            om["relayout_gbs"] = g
            om["relayout_frac_hbm"] = None if g is None else g / peaks["hbm_gbs"]
            om["relayout_l2"] = how
            del ost
            torch.cuda.empty_cache()
            per[ow.name] = om
        line["per_config"] = per
    if not args.no_per_config:   # the scan's bandwidth at scale (every workload's scan is <= 512 KB)
        sw = scan_bandwidth(device)
        sw["frac_hbm"] = sw["gbs"] / peaks["hbm_gbs"]
        line["scan_2e28"] = sw
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
