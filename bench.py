"""W12 GEMM benchmark on GB300.

Metric: W12 GEMM weight-GB/s (bytes of packed W12 weights streamed per second)
and the fraction of the HBM roofline, on the four GEMMs of a 27B-class dense
decoder layer (QKV 5120->7168, O 5120->5120, gate/up 5120->34816,
down 17408->5120).

One step = the four layer GEMMs at each of M = 1, 2, 4, 8: four independent
requests, each a chain of its four layer GEMMs (16 w12_gemm calls; a request's
chain runs in order on its own stream, every GEMM's grid capped at half the
SMs so that two requests' GEMMs share the GPU; STEP_FORM).  The same GEMMs as one chain on one stream, and as one
w12_gemm_list call, each GEMM reading its activations after the previous one
has completed, are timed beside it.  Weights resident in HBM as W12,
synthetic BF16 activations.  The per-step working set (4 x 496 MB of W12) is
larger than the 129 MB L2.  The four requests share the four layer tensors;
in the one-stream chain every tensor is re-read only after at least 228 MB of
other weights have passed through L2, and in the four-stream step the same
step with a distinct encoded copy of the layers per request measured 0.4151
against 0.4141 ms (0.2%): the requests' GEMMs of one layer do not serve each
other's weights from L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Prints one JSON line (rank 0).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_VALUES = (1, 2, 4, 8)
# the form of the timed step: "calls" (16 w12_gemm calls, one stream per
# request, each request's chain by programmatic dependent launch) or "list"
# (one w12_gemm_list call)
STEP_FORM = "calls"
SWEEP_M = (16, 24, 32, 63, 64, 128, 256)  # tree / batch verification rows
METRIC = "W12 GEMM weight-GB/s & % HBM roofline at M=1/16/64 (27B-class layers)"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1940.8)), "measured"
    return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bit_weight_02_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.startswith("w12_gemm_mma") or fn in ("w12_device.cuh", "w12_stream.cuh"):
            h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(shape_bytes):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_mma_dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    ratio = d.get("traffic_over_algorithmic")
    return None if ratio is None else ratio * shape_bytes


def tc_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bit_weight_02_gb300", "csrc")
    for fn in ("w12_gemm_tc.cu", "w12_device.cuh", "w12_stream.cuh"):
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def tensor_pipe_share():
    """sm__pipe_tensor_cycles_active (% of peak) of the tcgen05 kernel at
    M = 64 from the committed ncu summary, if it was taken on the current
    kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_tc_tensor_pipe.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != tc_source_hash():
        return None
    return d.get("tensor_pipe_active_pct")


# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_time_ms(local_ms: float, ws_n: int, device) -> float:
    """The whole job's time for the timed region: the slowest rank's (every
    rank runs the same units, so the job ends when the last one does)."""
    if ws_n <= 1:
        return local_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step: float, steps: int, ws_n: int, total_ms: float) -> float:
    """Whole-job throughput in GB/s: every rank streams bytes_per_step per step."""
    return bytes_per_step * steps * ws_n / (total_ms * 1e-3) / 1e9


def algorithmic_bytes(t, M: int) -> int:
    """W12 bytes + activations read + outputs written."""
    return t.nbytes() + 2 * M * t.K + 2 * M * t.N


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import lossless_bit_weight_02_gb300 as w12
    from lossless_bit_weight_02_gb300 import synth

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, bf16_peak, peak_src = peaks()

    # ---- resident W12 layer (encoded and verified on the GPU) ----
    layers = []
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES):
        Wd = synth.dense_weights_device(N, K, seed=1000 + i, device=dev)
        t = w12.w12_encode(Wd)
        st, nm = w12.w12_verify_roundtrip(Wd, t)
        assert st == w12.W12_OK, (name, st, nm)
        del Wd
        layers.append((name, t))
    torch.cuda.empty_cache()
    Ms = sorted(set(M_VALUES) | set(SWEEP_M))
    acts = {(M, name): synth.activations_device(M, t.K, seed=2000 + 10 * M + i, device=dev)
            for M in Ms for i, (name, t) in enumerate(layers)}
    outs = {(M, name): torch.empty(M, t.N, dtype=torch.bfloat16, device=dev)
            for M in Ms for name, t in layers}
    wsp = w12.Workspace(dev, max(w12.w12_gemm_workspace_bytes(M, t.N, t.K) for M in Ms for _, t in layers))
    stream = torch.cuda.current_stream(dev)
    wsp.ensure(max([w12.w12_gemm_workspace_bytes(M, t.N, t.K) for M in Ms for _, t in layers] +
                   [w12.w12_gemm_workspace_bytes(16, t.N, t.K, w12.make_opts(path=w12.W12_PATH_TC))
                    for _, t in layers]))
    # weights are resident and never written while the step runs, so every
    # GEMM may overlap the previous one (programmatic dependent launch)
    overlap = w12.make_opts(flags=w12.W12_GEMM_OVERLAP_PREVIOUS)
    calls = {(M, name): w12.GemmCall(acts[(M, name)], t, outs[(M, name)], wsp, stream=stream, opts=overlap)
             for M in Ms for name, t in layers}

    def calls_step(ev=None, m_values=M_VALUES):
        """The 16 w12_gemm calls as one chain on one stream (programmatic dependent launch)."""
        j = 0
        for M in m_values:
            for name, t in layers:
                if ev is not None:
                    ev[j][0].record(stream)
                calls[(M, name)]()
                if ev is not None:
                    ev[j][1].record(stream)
                j += 1

    # The step as four requests on four streams: request j's four layer GEMMs
    # run as a chain on stream j (programmatic dependent launch inside it, a
    # workspace of its own), so a GEMM of one request can take over the SMs
    # another request's GEMM is draining.  The streams fork from and join back
    # into `stream` every step, so events on `stream` bracket whole steps.
    # Each GEMM's grid is capped at half the SMs (max_ctas; the result is
    # bitwise the same on every grid), so two requests' GEMMs run side by side
    # and each one's start and tail overlap the other's work; these launches
    # go without programmatic dependent launch, which let a request's next
    # GEMM make its blocks resident early and hold SMs that another request's
    # GEMM could use (4.78-4.95 TB/s, depending on what had run before).
    # Measured on a GB300 (TB/s), caps without that overlap: 64: 4.73, 72: 4.85,
    # 76: 5.05, 80: 5.07, 88: 5.03; the full grid with it: 4.81 (reported
    # beside the headline as `calls_full_grid`).
    ws_bytes = max(w12.w12_gemm_workspace_bytes(M, t.N, t.K) for M in M_VALUES for _, t in layers)
    half_grid = max(1, torch.cuda.get_device_properties(dev).multi_processor_count // 2)

    class RequestStreams:
        def __init__(self, main, a_of, o_of, max_ctas=half_grid):
            self.main = main
            self.streams = [torch.cuda.Stream(dev) for _ in M_VALUES]
            self.fork = torch.cuda.Event()
            self.joins = [torch.cuda.Event() for _ in M_VALUES]
            # one workspace per request: its chain's GEMMs run one after another
            self.ws = [w12.Workspace(dev, ws_bytes) for _ in M_VALUES]
            flags = 0 if max_ctas else w12.W12_GEMM_OVERLAP_PREVIOUS
            opts = w12.make_opts(max_ctas=max_ctas, flags=flags)
            self.calls = [[w12.GemmCall(a_of[(M, name)], t, o_of[(M, name)], ws, stream=st, opts=opts)
                           for name, t in layers]
                          for M, st, ws in zip(M_VALUES, self.streams, self.ws)]

        def __call__(self):
            self.fork.record(self.main)
            for st in self.streams:
                st.wait_event(self.fork)
            # enqueued layer by layer across the requests' streams (0.3% faster
            # on a GB300 than request by request; stream priorities were slower)
            for li in range(len(layers)):
                for chain in self.calls:
                    chain[li]()
            for st, ev in zip(self.streams, self.joins):
                ev.record(st)
                self.main.wait_event(ev)

    streams_step = RequestStreams(stream, acts, outs)
    full_grid_step = RequestStreams(stream, acts, outs, max_ctas=0)

    # The step as w12_gemm_list calls: each list holds two requests' layer
    # GEMMs in one persistent launch, every GEMM reading its activations only
    # after its request's GEMM before it has completed (the dependency a chain
    # of layer GEMMs has).  The items go layer by layer with the two requests
    # side by side, so each depends on the item two places back and the items
    # a warp moves on to are seldom still waiting.  The two lists run on two
    # streams with their grids capped at half the SMs, as the calls do
    # (measured on a GB300: 4.78 TB/s against 4.39 for all four requests in one
    # full-grid list, and 4.21 for that list request by request).
    step_keys = [(M, name) for M in M_VALUES for name, _ in layers]
    tensor_of = dict(layers)
    list_pairs = [(M_VALUES[0], M_VALUES[3]), (M_VALUES[1], M_VALUES[2])]

    class PairLists:
        def __init__(self, main, a_of, o_of):
            self.main = main
            self.streams = [torch.cuda.Stream(dev) for _ in list_pairs]
            self.fork = torch.cuda.Event()
            self.joins = [torch.cuda.Event() for _ in list_pairs]
            opts = w12.make_opts(max_ctas=half_grid)
            self.calls = []
            for pr, st in zip(list_pairs, self.streams):
                keys = [(M, name) for name, _ in layers for M in pr]
                r = len(pr)
                self.calls.append(w12.GemmListCall([(a_of[k], tensor_of[k[1]], o_of[k], j - r if j >= r else -1, 0)
                                                    for j, k in enumerate(keys)], w12.Workspace(dev), opts=opts,
                                                   stream=st))

        def __call__(self):
            self.fork.record(self.main)
            for st in self.streams:
                st.wait_event(self.fork)
            for c in self.calls:
                c()
            for st, ev in zip(self.streams, self.joins):
                ev.record(st)
                self.main.wait_event(ev)

    list_call = PairLists(stream, acts, outs)

    # Both forms of the step are timed over the same number of steps; the
    # headline `value` is STEP_FORM's, the other is reported beside it.
    forms = {"calls": (streams_step, len(step_keys), "k_gemm_mma<1> (w12_gemm, M<=8)",
                       "16 w12_gemm calls: each request's (M's) four layer GEMMs in order on a stream of its "
                       f"own, the four requests' streams concurrent, every GEMM's grid capped at half the SMs "
                       f"(max_ctas {half_grid}) so two requests' GEMMs share the GPU"),
             "list": (list_call, len(list_pairs), "k_gemm_mma_list<1> (w12_gemm_list, M<=8)",
                      f"two w12_gemm_list calls on two streams, each over two requests' layer GEMMs (M pairs "
                      f"{list_pairs}) listed layer by layer with the two requests side by side, grids capped at "
                      f"half the SMs; each of a request's later layers reads its activations after the request's "
                      f"GEMM before it has completed")}
    other_form = "list" if STEP_FORM == "calls" else "calls"
    one_step, launches_per_step, step_kernel, step_note = forms[STEP_FORM]
    other_step = forms[other_form][0]
    step_bytes = sum(t.nbytes() for _, t in layers) * len(M_VALUES)
    alg_bytes = {(M, name): algorithmic_bytes(t, M) for M in Ms for name, t in layers}

    for _ in range(args.warmup):
        one_step()
        other_step()
        full_grid_step()
    torch.cuda.synchronize()
    # the list's outputs are bitwise those of the 16 separate calls
    list_out = {k: outs[k].clone() for k in step_keys}
    list_call()
    torch.cuda.synchronize()
    list_matches_calls = all(torch.equal(list_out[k].view(torch.int16), outs[k].view(torch.int16))
                             for k in step_keys)

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        one_step()
    stop.record(stream)
    torch.cuda.synchronize()
    if ws_n > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = job_time_ms(start.elapsed_time(stop), ws_n, dev)

    # The other form of the step, timed the same way after the timed region.
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for k in range(args.steps):
        other_step()
    c1.record(stream)
    torch.cuda.synchronize()
    other_ms = c0.elapsed_time(c1) / args.steps
    # ... and the 16 calls as one chain on one stream (every GEMM after the one
    # before it, the four requests serialised)
    c0.record(stream)
    for k in range(args.steps):
        calls_step()
    c1.record(stream)
    torch.cuda.synchronize()
    chain_ms = c0.elapsed_time(c1) / args.steps
    # ... and the four streams with every GEMM on the full grid
    c0.record(stream)
    for k in range(args.steps):
        full_grid_step()
    c1.record(stream)
    torch.cuda.synchronize()
    full_grid_ms = c0.elapsed_time(c1) / args.steps

    # Per-launch events of the 16-call step on 10 more steps: an event
    # between two launches keeps the second from overlapping the first, so
    # these launches run serialised (each pays its own fill and drain).
    n_ev = 10
    n_calls = len(step_keys)
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
            for _ in range(n_calls)] for _ in range(n_ev)]
    for k in range(n_ev):
        calls_step(evs[k])
    torch.cuda.synchronize()

    # run-to-run spread of the same step: 5 more batches of 50 steps, events
    # around each batch only (not part of `value`)
    batch_ms = []
    for _ in range(5):
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(50):
            one_step()
        b1.record(stream)
        torch.cuda.synchronize()
        batch_ms.append(b0.elapsed_time(b1) / 50)
    batch_ms.sort()
    noise = {"batches": 5, "steps_per_batch": 50,
             "gbs": [round(step_bytes / (x * 1e-3) / 1e9, 1) for x in batch_ms[::-1]],
             "spread_pct": round(100.0 * (batch_ms[-1] - batch_ms[0]) / statistics.median(batch_ms), 2)}

    # the same step replayed from a CUDA graph (how a serving engine launches a
    # fixed sequence of GEMMs): 10 steps per graph, on a side stream
    gstream = torch.cuda.Stream(dev)
    if STEP_FORM == "list":
        gcalls = [PairLists(gstream, acts, outs)]  # the streams fork from and join the capture stream
    else:
        gcalls = [RequestStreams(gstream, acts, outs)]  # the streams fork from and join the capture stream
    with torch.cuda.stream(gstream):
        for c in gcalls:
            c()
    torch.cuda.synchronize()
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=gstream):
        for _ in range(10):
            for c in gcalls:
                c()
    g_reps = max(3, args.steps // 10)
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gstream):
        step_graph.replay()
        ga.record(gstream)
        for _ in range(g_reps):
            step_graph.replay()
        gb.record(gstream)
    torch.cuda.synchronize()
    graph_ms = job_time_ms(ga.elapsed_time(gb), ws_n, dev)
    value_graph = job_value(step_bytes, 10 * g_reps, ws_n, graph_ms)
    del step_graph, gcalls

    # per-launch kernel durations (serialised launches of the 16-call step) -> per (M, layer)
    dur = {}
    j = 0
    for M in M_VALUES:
        for name, _ in layers:
            dur[(M, name)] = [evs[k][j][0].elapsed_time(evs[k][j][1]) for k in range(n_ev)]
            j += 1
    kern_ms = sum(sum(v) for v in dur.values())
    kern_bytes = sum(alg_bytes[key] * len(v) for key, v in dur.items())
    achieved_serial = kern_bytes / (kern_ms * 1e-3) / 1e9
    # The step's only kernel is k_gemm_mma<1> (16 launches that overlap:
    # programmatic dependent launch inside a request's chain, the requests'
    # streams side by side) or k_gemm_mma_list<1> (one launch), so
    # the kernel's device time per step is the step's device time, and the
    # roofline's achieved rate is the step's algorithmic bytes over it.
    step_alg_bytes = sum(alg_bytes[(M, n)] for M in M_VALUES for n, _ in layers)
    step_ms = total_ms / args.steps
    achieved = step_alg_bytes / (step_ms * 1e-3) / 1e9
    per_m = {}
    for M in M_VALUES:
        b = sum(layers_t.nbytes() for _, layers_t in layers)
        ms = sum(statistics.median(dur[(M, name)]) for name, _ in layers)
        per_m[str(M)] = {"weight_gbs": round(b / (ms * 1e-3) / 1e9, 1),
                         "roofline_frac": round(sum(alg_bytes[(M, n)] for n, _ in layers) / (ms * 1e-3) / 1e9
                                                / hbm_peak, 4)}
    per_layer = {name: round(statistics.median(dur[(1, name)]) * 1e3, 2) for name, _ in layers}

    # ---- M = 16..256 (tree / batch verification) ----
    # roofline per M: max(algorithmic bytes / HBM peak, 2MNK / BF16 peak)
    # The four layers run back to back (programmatic dependent launch), as in
    # the step; events bracket blocks of 6 passes, so no event sits between
    # two launches.  A short device sleep before the first event lets the
    # host queue the block's launches first.  The layers' 496 MB of W12 cycle
    # through the 129 MB L2.
    # `us_launch_events` is the sum of per-launch event intervals instead:
    # each launch then pays its own fill, drain and event overhead.
    def sweep_point(M, call_of):
        ev2 = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
               for _ in range(len(layers))]
        for _ in range(max(3, args.warmup)):
            for name, _ in layers:
                call_of(name)()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(200_000)  # ~0.1 ms of device time
            e0.record(stream)
            for _ in range(6):
                for name, _ in layers:
                    call_of(name)()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 6)
        ms = statistics.median(ts)
        tl = []
        per_layer = {name: [] for name, _ in layers}
        for _ in range(10):
            for j, (name, _) in enumerate(layers):
                ev2[j][0].record(stream)
                call_of(name)()
                ev2[j][1].record(stream)
            torch.cuda.synchronize()
            tl.append(sum(e[0].elapsed_time(e[1]) for e in ev2))
            for j, (name, _) in enumerate(layers):
                per_layer[name].append(ev2[j][0].elapsed_time(ev2[j][1]))
        b = sum(t.nbytes() for _, t in layers)
        ab = sum(alg_bytes[(M, n)] for n, _ in layers)
        flops = sum(2.0 * M * t.N * t.K for _, t in layers)
        floor_s = max(ab / (hbm_peak * 1e9), flops / (bf16_peak * 1e12))
        return {"weight_gbs": round(b / (ms * 1e-3) / 1e9, 1), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                "roofline_frac": round(floor_s / (ms * 1e-3), 4), "us": round(ms * 1e3, 1),
                "us_launch_events": round(statistics.median(tl) * 1e3, 1),
                "us_launch_events_per_layer": {n: round(statistics.median(v) * 1e3, 1) for n, v in per_layer.items()}}

    sweep = {"1": sweep_point(1, lambda name: calls[(1, name)])}
    sweep["1"]["path"] = "mma"
    for M in SWEEP_M:
        sweep[str(M)] = sweep_point(M, lambda name, M=M: calls[(M, name)])
        sweep[str(M)]["path"] = "mma" if M <= 16 else "tcgen05"
    tc16 = {name: w12.GemmCall(acts[(16, name)], t, outs[(16, name)], wsp, stream=stream,
                               opts=w12.make_opts(path=w12.W12_PATH_TC, flags=w12.W12_GEMM_OVERLAP_PREVIOUS))
            for name, t in layers}
    sweep["16_tcgen05"] = sweep_point(16, lambda name: tc16[name])
    sweep["16_tcgen05"]["path"] = "tcgen05"

    # ---- end to end through the public API with host buffers ----
    # Every step copies all of its activations host -> device in one copy (from
    # pinned memory), runs the 16 GEMMs through the public call (in the device
    # step's form), and reads all the outputs back in one copy.  As a serving
    # loop does, the device buffers are doubled and the copies have streams of
    # their own: step k+1's inputs go up while step k computes, and step k's
    # outputs come down while step k+1 computes (events keep each buffer pair
    # from being reused before its last step's copy is done).
    keys = [(M, name) for M in M_VALUES for name, _ in layers]
    align = lambda n: (n + 7) // 8 * 8  # 16-byte aligned views
    in_off, out_off, n_in, n_out = {}, {}, 0, 0
    for key in keys:
        in_off[key], n_in = n_in, n_in + align(acts[key].numel())
        out_off[key], n_out = n_out, n_out + align(outs[key].numel())
    h_in_all = torch.zeros(n_in, dtype=torch.bfloat16).pin_memory()
    for key in keys:
        h_in_all[in_off[key]:in_off[key] + acts[key].numel()].copy_(acts[key].reshape(-1).cpu())
    h_out_all = torch.empty(n_out, dtype=torch.bfloat16).pin_memory()
    e2e_sets = []
    for b in range(2):
        d_in_all = torch.empty(n_in, dtype=torch.bfloat16, device=dev)
        d_out_all = torch.empty(n_out, dtype=torch.bfloat16, device=dev)
        e2e_a, e2e_o = {}, {}
        for key in keys:
            a, o = acts[key], outs[key]
            e2e_a[key] = d_in_all[in_off[key]:in_off[key] + a.numel()].view(a.shape)
            e2e_o[key] = d_out_all[out_off[key]:out_off[key] + o.numel()].view(o.shape)
        if STEP_FORM == "list":
            call = PairLists(stream, e2e_a, e2e_o)
        else:
            call = RequestStreams(stream, e2e_a, e2e_o)
        e2e_sets.append((d_in_all, d_out_all, call))
    h2d = sum(acts[key].numel() * 2 for key in keys)
    d2h = sum(outs[key].numel() * 2 for key in keys)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # per buffer pair: inputs landed, step computed, outputs read
    landed = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):
        computed[b].record(stream)
        read[b].record(stream)

    def e2e_step(k):
        b = k % 2
        d_in, d_out, call = e2e_sets[b]
        up.wait_event(computed[b])  # step k-2, which read these inputs, has computed
        with torch.cuda.stream(up):
            d_in.copy_(h_in_all, non_blocking=True)
        landed[b].record(up)
        stream.wait_event(landed[b])
        stream.wait_event(read[b])  # step k-2's outputs have been read back
        call()
        computed[b].record(stream)
        down.wait_event(computed[b])
        with torch.cuda.stream(down):
            h_out_all.copy_(d_out, non_blocking=True)
        read[b].record(down)

    e2e_steps = max(10, min(args.steps, 500))
    for k in range(4):
        e2e_step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(e2e_steps):
        e2e_step(k)
    # the end waits for the last step's read-back
    stream.wait_event(read[(e2e_steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    # the outputs read back equal the device step's, bit for bit (same inputs, fixed order)
    e2e_match = all(torch.equal(h_out_all[out_off[key]:out_off[key] + outs[key].numel()].view(outs[key].shape),
                                outs[key].cpu()) for key in keys)

    # ---- the nested 8-bit view (W12_GEMM_NESTED8): the same GEMMs reading the hi plane only ----
    nested = {}
    for M in (1, 16, 64):
        row = {}
        for label, flags in (("exact", w12.W12_GEMM_OVERLAP_PREVIOUS),
                             ("nested8", w12.W12_GEMM_OVERLAP_PREVIOUS | w12.W12_GEMM_NESTED8)):
            o = w12.make_opts(flags=flags)
            xs = {K: synth.activations_device(M, K, seed=5000 + M + K, device=dev) for _, _, K in synth.LAYER_SHAPES}
            ys = {N: torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _, N, _ in synth.LAYER_SHAPES}
            wsp.ensure(max(w12.w12_gemm_workspace_bytes(M, t.N, t.K, o) for _, t in layers))
            cs = [w12.GemmCall(xs[t.K], t, ys[t.N], wsp, stream=stream, opts=o) for _, t in layers]
            for c in cs:
                c()
            torch.cuda.synchronize()
            reps = 50
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                for c in cs:
                    c()
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / reps
            # bytes each pass must read: the hi plane (and the lo plane for the exact pass), bases,
            # group offsets, escapes, activations and outputs
            rd = sum(t.hi.numel() + (0 if label == "nested8" else t.lo.numel()) + t.base.numel() +
                     4 * t.esc_ptr.numel() + 4 * t.n_esc + 2 * M * t.K + 2 * M * t.N for _, t in layers)
            row[label] = {"us_per_4_layers": round(us, 2), "gbs_read": round(rd / (us * 1e-6) / 1e9, 1),
                          "roofline_frac": round(rd / (us * 1e-6) / 1e9 / hbm_peak, 4)}
            del cs, xs, ys
        row["speedup"] = round(row["exact"]["us_per_4_layers"] / row["nested8"]["us_per_4_layers"], 3)
        nested[str(M)] = row
    nested["note"] = ("four layer GEMMs per round, 50 rounds back to back (PDL on); nested8 reads the hi plane "
                      "only (1 B/weight vs 1.5)")

    # ---- codec throughput on the config-1 layer (rows a1-a5): encode, decode, verify ----
    codec = {}
    ev = lambda: torch.cuda.Event(enable_timing=True)
    def med_host(f, n=5):  # median host time (ms) of a synchronous call
        ts = []
        for _ in range(n):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            f()
            torch.cuda.synchronize()
            ts.append((time.perf_counter() - t0) * 1e3)
        return statistics.median(ts)

    enc_ms = enc_alloc_ms = dec_ms = ver_ms = 0.0
    enc_bytes = dec_bytes = ver_bytes = 0
    enc_layers = {}
    for i, (name, N, K) in enumerate(synth.LAYER_SHAPES):
        Wd = synth.dense_weights_device(N, K, seed=1000 + i, device=dev)
        t = w12.w12_encode(Wd)  # warm; sizes the escape array
        pre = w12.empty_tensor(N, K, max(1024, 2 * t.n_esc), dev)
        w12.w12_encode(Wd, out=pre)
        # into preallocated buffers (converting many layers), and allocating
        # its own (the call includes the one host sync for the escape count)
        e_ms = med_host(lambda: w12.w12_encode(Wd, out=pre))
        enc_alloc_ms += med_host(lambda: w12.w12_encode(Wd))
        enc_ms += e_ms
        b = 2 * 2 * N * K + t.nbytes()  # W read twice (window, pack) + W12 written
        enc_bytes += b
        enc_layers[name] = {"us": round(e_ms * 1e3, 1), "gbs": round(b / (e_ms * 1e-3) / 1e9, 1)}
        out = torch.empty_like(Wd)
        ds = []
        for _ in range(5):
            a, bb = ev(), ev()
            a.record(stream)
            w12.w12_decode(t, out)
            bb.record(stream)
            torch.cuda.synchronize()
            ds.append(a.elapsed_time(bb))
        dec_ms += statistics.median(ds)
        dec_bytes += t.nbytes() + 2 * N * K
        ver_ms += med_host(lambda: w12.w12_verify_roundtrip(Wd, t))
        ver_bytes += t.nbytes() + 2 * N * K
        assert w12.w12_verify_roundtrip(Wd, t) == (w12.W12_OK, 0)
        del Wd, out, pre
    codec = {"encode_gbs": round(enc_bytes / (enc_ms * 1e-3) / 1e9, 1),
             "encode_gbs_allocating": round(enc_bytes / (enc_alloc_ms * 1e-3) / 1e9, 1),
             "encode_per_layer": enc_layers,
             "decode_gbs": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
             "verify_gbs": round(ver_bytes / (ver_ms * 1e-3) / 1e9, 1),
             "note": "algorithmic bytes / time over the four layer tensors (encode: W read twice + W12 "
                     "written), medians of 5; encode (into preallocated buffers, or allocating its own) and "
                     "verify are host-synchronous calls timed on the host clock, decode by CUDA events"}
    torch.cuda.empty_cache()

    # ---- 64-layer stack (config 3): convert + load-time check, then stream ----
    stack = None
    if not args.no_stack:
        t_conv = time.perf_counter()
        stk = []
        for layer in range(64):
            for i, (name, N, K) in enumerate(synth.LAYER_SHAPES):
                Wd = synth.dense_weights_device(N, K, seed=3000 + 16 * layer + i, device=dev)
                t = w12.w12_encode(Wd)
                st, nm = w12.w12_verify_roundtrip(Wd, t)
                assert st == w12.W12_OK, (layer, name, st, nm)
                del Wd
                stk.append(t)
        torch.cuda.synchronize()
        conv_s = time.perf_counter() - t_conv
        torch.cuda.empty_cache()
        sb = sum(t.nbytes() for t in stk)
        nw = sum(t.N * t.K for t in stk)
        stack = {"layers": 64, "tensors": len(stk), "w12_gb": round(sb / 1e9, 3), "bf16_gb": round(2 * nw / 1e9, 3),
                 "bits_per_weight": round(8 * sb / nw, 4),
                 "convert_and_verify_s": round(conv_s, 2)}
        for M in (1, 16):
            acts_s = {K: synth.activations_device(M, K, seed=M * 100 + K, device=dev) for _, _, K in synth.LAYER_SHAPES}
            outs_s = {N: torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _, N, _ in synth.LAYER_SHAPES}
            wsp.ensure(max(w12.w12_gemm_workspace_bytes(M, t.N, t.K) for t in stk[:4]))
            cs = [w12.GemmCall(acts_s[t.K], t, outs_s[t.N], wsp, stream=stream, opts=overlap) for t in stk]
            for c in cs:
                c()
            torch.cuda.synchronize()
            a, b = ev(), ev()
            reps = 5
            a.record(stream)
            for _ in range(reps):
                for c in cs:
                    c()
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            stack[f"m{M}"] = {"pass_ms": round(ms, 3), "weight_gbs": round(sb / (ms * 1e-3) / 1e9, 1),
                              "roofline_frac": round(sum(algorithmic_bytes(t, M) for t in stk) / (ms * 1e-3) / 1e9
                                                     / hbm_peak, 4)}
            # the same 256 launches captured once in a CUDA graph (on a side
            # stream: capture needs one) and replayed
            gs = torch.cuda.Stream(dev)
            gcs = [w12.GemmCall(acts_s[t.K], t, outs_s[t.N], wsp, stream=gs, opts=overlap) for t in stk]
            torch.cuda.synchronize()
            with torch.cuda.stream(gs):
                for c in gcs:  # fills the launch caches before capture
                    c()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                for c in gcs:
                    c()
            with torch.cuda.stream(gs):
                graph.replay()
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(gs)
            with torch.cuda.stream(gs):
                for _ in range(reps):
                    graph.replay()
            b.record(gs)
            torch.cuda.synchronize()
            gms = a.elapsed_time(b) / reps
            stack[f"m{M}"]["graph"] = {"pass_ms": round(gms, 3), "weight_gbs": round(sb / (gms * 1e-3) / 1e9, 1)}
            del graph, gcs
            # The stack as one dependent chain through w12_gemm_list (256
            # GEMMs, four launches of 64): per layer, QKV reads the layer
            # input; O reads a fixed stand-in for the attention output and
            # waits for QKV; gate/up reads O's output and writes silu(g) * u
            # (W12_GEMM_SILU_MUL); down reads that and writes the next
            # layer's input.
            xs = [synth.activations_device(M, 5120, seed=M * 100 + 7, device=dev),
                  torch.empty(M, 5120, dtype=torch.bfloat16, device=dev)]
            attn = synth.activations_device(M, 5120, seed=M * 100 + 8, device=dev)
            qb = torch.empty(M, 7168, dtype=torch.bfloat16, device=dev)
            hb = torch.empty(M, 5120, dtype=torch.bfloat16, device=dev)
            ab = torch.empty(M, 17408, dtype=torch.bfloat16, device=dev)
            chain = []
            for layer in range(64):
                tq, to, tg, td = stk[4 * layer:4 * layer + 4]
                j = len(chain)
                chain += [(xs[layer % 2], tq, qb, j - 1, 0), (attn, to, hb, j, 0),
                          (hb, tg, ab, j + 1, w12.W12_GEMM_SILU_MUL), (ab, td, xs[(layer + 1) % 2], j + 2, 0)]
            lc = w12.GemmListCall(chain, w12.Workspace(dev), stream=stream)
            lc()
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(stream)
            for _ in range(reps):
                lc()
            b.record(stream)
            torch.cuda.synchronize()
            lms = a.elapsed_time(b) / reps
            stack[f"m{M}"]["list_chain"] = {
                "pass_ms": round(lms, 3), "weight_gbs": round(sb / (lms * 1e-3) / 1e9, 1),
                "roofline_frac": round(sum(algorithmic_bytes(t, M) for t in stk) / (lms * 1e-3) / 1e9 / hbm_peak, 4),
                "launches": (len(chain) + w12.W12_LIST_MAX - 1) // w12.W12_LIST_MAX,
                "note": "256 GEMMs as a dependent chain (each layer: QKV; O after QKV; gate/up with the fused "
                        "silu(g)*u epilogue after O; down after gate/up; next layer's QKV after down), "
                        "w12_gemm_list"}
            del lc, chain, xs, attn, qb, hb, ab
        del stk
        torch.cuda.empty_cache()

    # ---- best-first draft-tree node selection (the next row after the GEMM) ----
    tree = tree_bench(dev, cpu=(rank == 0 and not args.no_cpu_baseline))
    gdn = gdn_bench(dev, cpu=(rank == 0 and not args.no_cpu_baseline), hbm_peak=hbm_peak)

    # ---- what a plain device copy reaches at these sizes (context for the roofline) ----
    # MEASURED_PEAKS' HBM figure is a 2 GiB copy; a copy of one layer's W12 bytes
    # pays the same launch, ramp-up and tail costs that a single GEMM launch does.
    size_cal = {}
    flush_c = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for name, t in layers:
        nb = t.nbytes()
        src = torch.empty(nb, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        best = None
        for _ in range(8):
            flush_c.zero_()
            a, b = ev(), ev()
            a.record(stream)
            dst.copy_(src)
            b.record(stream)
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        size_cal[name] = {"w12_mb": round(nb / 1e6, 1), "copy_gbs": round(2 * nb / (best * 1e-3) / 1e9, 1)}
        del src, dst
    del flush_c
    torch.cuda.empty_cache()
    size_cal["method"] = ("torch dst.copy_(src) of the layer's W12 byte count, read+write bytes / best of 8, "
                          "L2 flushed before each copy")

    # the metric's three points, M = 1 / 16 / 64, each the four layers back to
    # back (the sweep's method); M = 64 runs on the tcgen05 path
    roofline_by_m = {}
    for M in (1, 16, 64):
        sp = sweep[str(M)]
        roofline_by_m[str(M)] = {"frac": sp["roofline_frac"], "weight_gbs": sp["weight_gbs"],
                                 "tflops": sp["tflops"], "us_4_layers": sp["us"], "path": sp["path"],
                                 "bound": "hbm" if M < 200 else "hbm+tensor"}
    tp = tensor_pipe_share()
    if tp is not None:
        roofline_by_m["64"]["tensor_pipe_active_pct_ncu"] = tp

    value = job_value(step_bytes, args.steps, ws_n, total_ms)
    e2e_val = step_bytes * e2e_steps * ws_n / (e2e_ms * 1e-3) / 1e9
    top_bytes = sum(alg_bytes[(M, n)] for M in M_VALUES for n, _ in layers) / launches_per_step
    traffic = ncu_traffic(top_bytes)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian weights with LogNormal(0,0.5) channel scale, 0.1% zeros, "
                "0.05% x2^9 outliers; N(0,1) activations)",
        "config": {"workload": "27B-class decoder layer GEMMs (QKV 7168x5120, O 5120x5120, gate/up "
                               "34816x5120, down 5120x17408), M in {1,2,4,8}, W12 weights resident",
                   "global_batch": list(M_VALUES), "parallelism": f"replica x{ws_n} (N-sharding not needed)",
                   "grid": f"each GEMM of the step capped at {half_grid} CTAs (half the SMs; max_ctas), "
                           "four request streams, no programmatic dependent launch",
                   "l2": "inputs larger than L2 (4 x 496 MB W12 per step; the requests share the layer tensors, "
                         "and distinct copies per request measured 0.2% slower: no reuse through L2)",
                   "bits_per_weight": round(sum(t.nbytes() for _, t in layers) * 8 /
                                            sum(t.N * t.K for _, t in layers), 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "kernel": step_kernel,
                     "method": "algorithmic bytes of the step's 16 GEMMs (W12 bytes + activations + "
                               "outputs) / the step's device time in the timed region (the step's only "
                               "kernel; its launches overlap)",
                     "bytes_per_step": step_alg_bytes,
                     "serialised_launches": {
                         "achieved": round(achieved_serial, 1), "frac": round(achieved_serial / hbm_peak, 4),
                         "steps": n_ev, "kernel": "k_gemm_mma<1> (w12_gemm)",
                         "note": "the step as 16 w12_gemm calls with CUDA events around every launch, 10 steps "
                                 "after the timed region; an event between launches serialises them, so each "
                                 "pays its own fill and drain"}},
        "step_form": {"headline": STEP_FORM, "note": step_note,
                      other_form: {"value": round(step_bytes / (other_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                                   "ms_per_step": round(other_ms, 4), "note": forms[other_form][3]},
                      "one_stream_chain": {"value": round(step_bytes / (chain_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                                           "ms_per_step": round(chain_ms, 4),
                                           "note": "the 16 w12_gemm calls as one chain on one stream (every GEMM "
                                                   "after the one before it, the requests serialised)"},
                      "calls_full_grid": {"value": round(step_bytes / (full_grid_ms * 1e-3) / 1e9, 1),
                                          "unit": "GB/s", "ms_per_step": round(full_grid_ms, 4),
                                          "note": "the four request streams with every GEMM on the full grid, "
                                                  "chained by programmatic dependent launch"},
                      "list_matches_calls_bitwise": list_matches_calls},
        "roofline_by_m": roofline_by_m,
        "value_graph": {"value": round(value_graph, 1), "unit": "GB/s",
                        "note": "the same step replayed from a CUDA graph (10 steps per graph)"},
        "per_m": per_m, "per_layer_us_m1": per_layer, "sweep": sweep, "codec": codec, "stack": stack,
        "tree": tree,
        "gdn": gdn,
        "noise": noise,
        "size_calibration": size_cal, "nested8": nested,
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "matches_device_outputs": e2e_match,
                "method": "per step: one pinned host->device copy of all 16 activations, the step's GEMMs "
                          f"({step_note}), one device->host copy of all outputs; two device buffer pairs and "
                          "copy streams of their own, so a step's copies overlap the neighbouring steps' GEMMs",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(layers, budget_s=args.cpu_seconds)
    if ws_n > 1:
        dist.destroy_process_group()
    return rank, result


# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle (decode + FP64 dot products, OpenMP over rows) on a bounded
    sample of the same workload: the first `rows` rows of each layer shape at
    M = 1, 2, 4, 8.  Encoding is done once per sample size, outside timing."""

    def __init__(self):
        import oracle
        from lossless_bit_weight_02_gb300 import synth
        oracle.build()
        self.oracle, self.synth = oracle, synth
        self.cache = {}

    def _prepared(self, rows):
        if rows not in self.cache:
            items = []
            for i, (name, N, K) in enumerate(self.synth.LAYER_SHAPES):
                st, ref = self.oracle.encode(self.synth.dense_weights(rows, K, seed=1000 + i))
                nb = ref.hi.size + ref.lo.size + rows + 4 * (rows + 1) + 6 * ref.n_esc
                for M in M_VALUES:
                    items.append((self.synth.activations(M, K, seed=2000 + 10 * M + i), ref, nb))
            self.cache[rows] = items
        return self.cache[rows]

    def run(self, rows):
        """One pass over the sample: (weight bytes, seconds)."""
        b, sec = 0.0, 0.0
        for A, ref, nb in self._prepared(rows):
            t0 = time.perf_counter()
            self.oracle.gemm(A, ref)
            sec += time.perf_counter() - t0
            b += nb
        return b, sec

    def rows_for(self, seconds):
        rows = 16
        while rows < 4096:
            b, s = self.run(rows)
            if s * 2 > seconds:
                break
            rows *= 2
        return rows


TREE_CASES = (  # (requests, positions, candidates, budget, shared)
    (1, 8, 8, 32, False),    # one request, 8-position lattice, 32 nodes
    (1, 16, 8, 63, False),   # 16 positions, 63 nodes
    (64, 8, 8, 32, False),   # a batch, 32 nodes per request
    (8, 16, 8, 256, True),   # a node budget shared by 8 requests
)


def tree_bench(dev, cpu: bool):
    """w12_tree_select on the pages' tree sizes (Dirichlet(0.3) log-probabilities):
    device time per call (CUDA events over 200 calls) and, beside it, the oracle."""
    import torch
    import lossless_bit_weight_02_gb300 as w12
    res = {}
    for R, D, C, B, shared in TREE_CASES:
        rng = np.random.default_rng(R * 100 + D)
        lp_h = np.log(rng.dirichlet(np.full(C, 0.3), size=(R, D))).astype(np.float32)
        lp = torch.from_numpy(lp_h).to(dev)
        call = w12.TreeCall(lp, B, shared)
        for _ in range(10):
            out = call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(200):
            call()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / 200
        kept = int(out["count"].sum())
        # device time without the host: 20 calls captured in a CUDA graph, replayed
        gs = torch.cuda.Stream(dev)
        gcall = w12.TreeCall(lp, B, shared, stream=gs)
        with torch.cuda.stream(gs):
            gcall()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(20):
                gcall()
        with torch.cuda.stream(gs):  # replays, and the events around them, on one stream
            graph.replay()
            torch.cuda.synchronize()
            a.record(gs)
            for _ in range(10):
                graph.replay()
            b.record(gs)
        torch.cuda.synchronize()
        g_us = a.elapsed_time(b) * 1e3 / 200
        row = {"us": round(us, 2), "us_graph": round(g_us, 2), "nodes": kept,
               "nodes_per_s": round(kept / (g_us * 1e-6), 1)}
        if cpu:
            from oracle import tree as tree_oracle
            t0 = time.perf_counter()
            n = 0
            while time.perf_counter() - t0 < 0.5:
                tree_oracle.select(lp_h, B, shared)
                n += 1
            row["oracle_us"] = round((time.perf_counter() - t0) * 1e6 / n, 1)
        res[f"R{R}_D{D}_C{C}_B{B}_{'shared' if shared else 'per_request'}"] = row
    res["note"] = ("GPU: one warp per request (best-first with first-child / next-sibling successors); a shared "
                   "budget adds a one-warp merge (and, if a short first-pass list runs out, a second pass). us: "
                   "eager calls back to back (host launch included); us_graph: the same calls replayed from a "
                   "CUDA graph (device time; nodes_per_s uses it). oracle_us: the Python oracle (test "
                   "infrastructure), one host thread")
    return res


GDN_CASES = (  # (requests, positions, candidates, node budget shared by the requests)
    (1, 16, 8, 63),
    (8, 16, 8, 256),
)


def gdn_trees(dev, R, Dp, C, B):
    """A best-first tree from w12_tree_select (Dirichlet(0.3) log-probabilities,
    `B` nodes shared by `R` requests of `Dp` positions): parent and req."""
    import torch
    import lossless_bit_weight_02_gb300 as w12
    rng = np.random.default_rng(700 + R)
    lp = torch.from_numpy(np.log(rng.dirichlet(np.full(C, 0.3), size=(R, Dp))).astype(np.float32)).to(dev)
    sel = w12.w12_tree_select(lp, B, True)
    n = int(sel["count"][0])
    return sel["parent"][:n].cpu().numpy().astype(np.int32), sel["req"][:n].cpu().numpy().astype(np.int32)


def gdn_bench(dev, cpu: bool, hbm_peak: float):
    """w12_gdn_tree on best-first trees (one GDN layer: 32 heads of 128):
    device time per call for the path and WY kernels, the HBM floor of the
    bytes the call must move, and the oracle beside it."""
    import torch
    import lossless_bit_weight_02_gb300 as w12
    from lossless_bit_weight_02_gb300 import synth
    H, D = synth.GDN_HEADS, synth.GDN_DIM
    res = {}
    for R, Dp, C, B in GDN_CASES:
        parent, req = gdn_trees(dev, R, Dp, C, B)
        n = len(parent)
        host = synth.gdn_inputs(n, H, D, seed=800 + R, R=R, parent=parent, req=req)
        S0, q, k, v, alpha, beta = host[:6]
        bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)  # noqa
        args = (t(S0), bf(q), bf(k), bf(v), t(alpha), t(beta), t(parent), t(req))
        # bytes a call must move at least: S0, q, k, v, alpha, beta, parent, req in; o out
        alg = S0.nbytes + q.nbytes + k.nbytes + v.nbytes + alpha.nbytes + beta.nbytes + 8 * n + n * H * D * 4
        row = {"nodes": n, "requests": R, "heads": H, "dim": D, "depth_max": int(max(
            len(_gdn_path_len(parent, i)) for i in range(n))), "bytes": alg,
               "floor_us": round(alg / (hbm_peak * 1e9) * 1e6, 2)}
        outs = {}
        for mode, name in ((w12.W12_GDN_PATH, "path"), (w12.W12_GDN_WY, "wy")):
            gs = torch.cuda.Stream(dev)
            call = w12.GdnCall(*args, mode=mode, stream=gs)
            with torch.cuda.stream(gs):
                for _ in range(5):
                    call()
            torch.cuda.synchronize()
            assert call.status() == w12.W12_OK
            outs[name] = call.out.clone()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(10):
                    call()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(gs):
                graph.replay()
                torch.cuda.synchronize()
                a.record(gs)
                for _ in range(20):
                    graph.replay()
                b.record(gs)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / 200
            row[name] = {"us_graph": round(us, 2), "nodes_per_s": round(n / (us * 1e-6), 1),
                         "roofline_frac": round(row["floor_us"] / us, 4)}
        d = (outs["wy"] - outs["path"]).abs()
        row["wy_vs_path_max_rel"] = float((d / outs["path"].abs().clamp_min(1e-3)).max())
        if cpu:
            from oracle import gdn as gdn_oracle
            f32 = lambda b: (np.asarray(b).astype(np.uint32) << 16).view(np.float32)  # noqa
            hs = 2  # a sample of heads; the oracle's time scales with the head count
            t0 = time.perf_counter()
            for r in range(R):
                idx = np.flatnonzero(req == r)
                remap = {int(j): x for x, j in enumerate(idx)}
                par = np.array([remap[int(parent[j])] if parent[j] >= 0 else -1 for j in idx], np.int64)
                gdn_oracle.path_outputs(S0[r, :hs], f32(q[idx, :hs]), f32(k[idx, :hs]), f32(v[idx, :hs]),
                                        alpha[idx, :hs], beta[idx, :hs], par)
            row["oracle_us"] = round((time.perf_counter() - t0) * 1e6 * H / hs, 1)
            row["oracle_sample"] = f"{hs} of {H} heads, scaled by {H // hs}"
        res[f"R{R}_B{B}"] = row
    res["note"] = ("Gated delta rule along every node's root path (hybrid-model tree verification), trees from "
                   "w12_tree_select; path: one CTA per (node, head), sequential rank-one updates; wy: keys and "
                   "queries times the root state on the tensor cores, then a warp per (node, head) solves its own "
                   "path's coefficients. "
                   "us_graph: CUDA-graph replay, device time per call. floor_us: the call's minimum bytes at "
                   "the measured HBM peak. oracle_us: the FP64 Python oracle (path definition), one host thread")
    return res


def _gdn_path_len(parent, i):
    path = []
    while i >= 0:
        path.append(i)
        i = int(parent[i])
    return path


def cpu_baseline(layers=None, budget_s=10.0):
    smp = OracleSample()
    rows = smp.rows_for(budget_s / 4)
    b = s = 0.0
    passes = 0
    while s < budget_s and passes < 64:
        db, ds = smp.run(rows)
        b += db
        s += ds
        passes += 1
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": smp.oracle.num_threads(), "kind": "oracle",
            "sample": f"oracle decode+FP64 GEMM on the first {rows} rows of each of the 4 layer shapes at "
                      f"M=1,2,4,8, {passes} passes, {s:.1f} s of CPU time"}


def run_reference(args):
    """The oracle timed as the reference arm, on the host cores."""
    ws_n, rank, local = dist_env()
    if rank != 0:
        return rank, None
    smp = OracleSample()
    step_s = min(args.ref_step_seconds, 150.0 / max(1, args.steps + args.warmup))
    rows = smp.rows_for(step_s)
    for _ in range(args.warmup):
        smp.run(rows)
    total_b = total_s = 0.0
    for _ in range(args.steps):
        b, s = smp.run(rows)
        total_b += b
        total_s += s
    v = total_b / total_s / 1e9
    threads = smp.oracle.num_threads()
    cb = {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
          "sample": f"per step: oracle decode+FP64 GEMM on the first {rows} rows of each layer shape at "
                    f"M=1,2,4,8"}
    return 0, {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "27B-class decoder layer GEMMs (QKV 7168x5120, O 5120x5120, "
                                                     "gate/up 34816x5120, down 5120x17408), M in {1,2,4,8}, "
                                                     "row sample on the CPU oracle"},
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_case(args):
    """One layer GEMM launched `iters` times (for profiler captures): prints
    the median kernel time and weight-GB/s, no JSON contract."""
    import torch

    import lossless_bit_weight_02_gb300 as w12
    from lossless_bit_weight_02_gb300 import synth

    if args.case == "tree":  # one best-first selection, `iters` times: --tree R D C B shared
        R, D, C, B, shared = args.tree
        rng = np.random.default_rng(R * 100 + D)
        lp = torch.from_numpy(np.log(rng.dirichlet(np.full(C, 0.3), size=(R, D))).astype(np.float32)).cuda()
        call = w12.TreeCall(lp, B, bool(shared))
        for _ in range(args.iters):
            out = call()
        torch.cuda.synchronize()
        print(f"case tree R={R} D={D} C={C} B={B} shared={shared}: {int(out['count'].sum())} nodes kept")
        return
    if args.case == "gdn":  # the 256-node, 8-request GDN tree, both kernels, `iters` times each
        R, Dp, C, B = GDN_CASES[-1]
        parent, req = gdn_trees(torch.device("cuda"), R, Dp, C, B)
        n, H, D = len(parent), synth.GDN_HEADS, synth.GDN_DIM
        host = synth.gdn_inputs(n, H, D, seed=800 + R, R=R, parent=parent, req=req)
        bf = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()  # noqa
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa
        dargs = (t(host[0]), bf(host[1]), bf(host[2]), bf(host[3]), t(host[4]), t(host[5]), t(parent), t(req))
        for mode in (w12.W12_GDN_PATH, w12.W12_GDN_WY):
            call = w12.GdnCall(*dargs, mode=mode)
            for _ in range(args.iters):
                call()
            torch.cuda.synchronize()
            assert call.status() == w12.W12_OK
        print(f"case gdn: {n} nodes, {R} requests, {H} heads of {D}: path and WY, {args.iters} calls each")
        return
    if args.case == "list":  # the bench step's 16 GEMMs as one w12_gemm_list call (its list form), `iters` times
        layers = []
        for i, (name, N, K) in enumerate(synth.LAYER_SHAPES):
            layers.append((name, w12.w12_encode(synth.dense_weights_device(N, K, seed=1000 + i))))
        keys = [(M, name) for name, _ in layers for M in M_VALUES]  # layer by layer, requests side by side
        tof = dict(layers)
        R = len(M_VALUES)
        entries = [(synth.activations_device(M, tof[n].K, seed=2000 + 10 * M + j), tof[n],
                    torch.empty(M, tof[n].N, dtype=torch.bfloat16, device="cuda"), j - R if j >= R else -1, 0)
                   for j, (M, n) in enumerate(keys)]
        call = w12.GemmListCall(entries, w12.Workspace("cuda"))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        call()
        e0.record()
        for _ in range(args.iters):
            call()
        e1.record()
        torch.cuda.synchronize()
        print(f"case list: 16 dependent GEMMs per call, {e0.elapsed_time(e1) * 1e3 / args.iters:.1f} us per call")
        return
    shapes = {name: (i, N, K) for i, (name, N, K) in enumerate(synth.LAYER_SHAPES)}
    i, N, K = shapes[args.case]
    Wd = synth.dense_weights_device(N, K, seed=1000 + i)
    t = w12.w12_encode(Wd)
    if args.codec:  # encode, decode and verify of the layer, `iters` times each
        out = torch.empty_like(Wd)
        for _ in range(args.iters):
            t = w12.w12_encode(Wd)
            w12.w12_decode(t, out)
            st, nm = w12.w12_verify_roundtrip(Wd, t)
            assert st == w12.W12_OK and nm == 0
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), Wd.view(torch.int16))
        print(f"case {args.case} codec: {args.iters} encode/decode/verify rounds, bit-exact")
        return
    del Wd
    A = synth.activations_device(args.m, K, seed=2000 + 10 * args.m + i)
    Y = torch.empty(args.m, N, dtype=torch.bfloat16, device="cuda")
    ws = w12.Workspace("cuda", w12.w12_gemm_workspace_bytes(args.m, N, K))
    call = w12.GemmCall(A, t, Y, ws)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    times = []
    for _ in range(args.iters):
        flush.zero_()  # evict the weights from L2 between launches
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    med = statistics.median(times)
    print(f"case {args.case} M={args.m}: {med * 1e3:.2f} us, {t.nbytes() / (med * 1e-3) / 1e9:.1f} weight-GB/s")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=5.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true", help="skip the 64-layer stack measurement")
    ap.add_argument("--case", default=None, help="profile one layer GEMM (qkv, o, gate_up, down), the step's GEMMs as one "
                    "w12_gemm_list chain (list), the tree selection (tree) or the GDN tree kernels (gdn)")
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--codec", action="store_true", help="with --case: encode, decode and verify the layer")
    ap.add_argument("--tree", type=int, nargs=5, default=(1, 8, 8, 32, 0), metavar=("R", "D", "C", "B", "SHARED"),
                    help="with --case tree: requests, positions, candidates, budget, shared (0/1)")
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        rank, res = run_reference(args)
    else:
        rank, res = run_gpu(args)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
