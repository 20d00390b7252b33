"""Benchmark of the deterministic W-way bf16 reduce on GB300.

Default workload: W = 8 bf16 partials of [32, 4096] (n = 131,072 elements,
256 KiB each; normal(0, 1), seed 1) -- the decode-sized message of the
one-shot all-reduce.  One step = one ``arx_reduce`` call: every element of
the 8 partials is read once, summed in fp32 in rank order and written once
as bf16.  Metric: HBM GB/s = (W + 1) * n * 2 bytes / time per call, and
microseconds per call.

Timing rules followed:
* inputs resident in HBM before the timed region; the calls rotate over
  enough buffer sets that their footprint is more than 3x the L2, so no call
  finds its inputs in L2 (stated in ``config``);
* >= 3 untimed warm-up steps, then exactly K timed steps, all launched from
  CUDA graphs (captured off the clock) on one stream; the timing events are
  recorded by the graphs themselves, the start one when the last of 64
  untimed lead-in calls completes and the end one when the last timed call
  completes (64 untimed calls follow), so the region holds exactly K call
  completions of a running stream of calls; L2 is flushed before the timed
  replay; a barrier and a device synchronise on both sides; the maximum over
  ranks is reported;
* nvidia-smi clocks and throttle reasons are sampled around the timed region.

Extra objects on the one JSON line: ``roofline`` (the reduce kernel against
the measured HBM copy bandwidth), ``cpu_baseline`` / ``cpu_baseline_1thread``
(the CPU oracle on all host cores and on one, bounded samples, timed in a
child process without CUDA), ``sweep`` (GB/s against size at W = 2, 4, 8),
``external_writer`` (a host thread raises the flags, the GPU reduces the
page-locked slots), ``e2e`` (the
same metric through ``arx_reduce_host`` with pinned host buffers, the
partials crossing the CPU-GPU link every call, against the link's measured
pinned copy rate), ``bandwidth`` (bandwidth-bound sizes: W=4 [1024, 8192] in
place, W=8 at 16 MiB and 256 MiB per partial), ``protocol`` (``arx_step``
per step in a captured graph, for each barrier variant), ``protocol_graph``
(10,000 steps with fresh partials captured in one CUDA graph), ``protocol_host_slots``
(the step with its slot banks in page-locked host memory), ``latency_floor``
(the same call with 1 KiB partials), ``hot_l2`` (inputs left in L2,
labelled), ``stream_launch`` (eager launches through the binding, no graph).

``--impl reference`` times the CPU oracle instead (the reference arm: there
is no reference implementation to install, the pages hold no code to build).
Multi-GPU (torchrun): every rank runs an independent replica of the
workload (the reduce has no cross-GPU step on one box); value = all ranks'
bytes / the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W-way bf16 reduce HBM GB/s ((W+1)·n·2 B / t); µs/call at bf16 [32,4096]"
DEFAULT_WORKLOAD = "w8_32x4096_normal"
FALLBACK_HBM_GBS = 6800.0
GRAPH_CALLS = 1000
QUEUE_AHEAD_CYCLES = 400_000   # ~0.2 ms at 2 GHz: longer than submitting a graph replay
LEAD_IN = 64                   # untimed calls at the head of the first timed graph (L2 turned over)
ROTATE_FACTOR = 3          # rotation footprint >= this many L2 sizes


# ---------------------------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by the gloo tests)

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate_over_ranks(elapsed_s: float, units: float) -> tuple[float, float]:
    """(max elapsed over ranks, sum of units over ranks); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_s, units
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def rotation_sets(set_bytes: int, l2_bytes: int, cap: int = 4096) -> int:
    """Buffer sets needed so that the rotation footprint exceeds ROTATE_FACTOR x L2."""
    need = (ROTATE_FACTOR * l2_bytes) // max(1, set_bytes) + 1
    return int(max(1, min(cap, need)))


def gbs(bytes_per_call: float, seconds_per_call: float) -> float:
    return bytes_per_call / seconds_per_call / 1e9


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh)
    except (OSError, ValueError):
        return {}


def kernel_source_hash() -> str:
    """Hash of the reduce kernel's sources: ties a stored ncu traffic figure to this code.

    Comments and whitespace are left out, so editing a comment keeps the
    figure; any change to the code itself gives a new hash.
    """
    h = hashlib.sha256()
    for rel in ("deterministic_shot_all_gb300/csrc/reduce.cu",
                "deterministic_shot_all_gb300/csrc/arx_device.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                  # line comments
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, n: int) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if taken on this
    kernel source at this size."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    e = rec.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    if e.get("n") is not None and int(e["n"]) != n:
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (index, SM MHz, max, reasons)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(ts=ts, sm=float(parts[2]), smax=float(parts[3]),
                                 power=float(parts[4]) if parts[4][:1].isdigit() else None,
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        window = [r for r in rows if self.t0 is not None and self.t0 - 0.15 <= r["ts"] <= (self.t1 or 0) + 0.15]
        used = window if window else rows
        reasons = set()
        for r in used:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in used),
                "sm_max_mhz": max(r["smax"] for r in used),
                "reasons": sorted(reasons),
                "samples_in_window": len(window), "samples": len(rows)}


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)

ORACLE_WARM_S = 1.0   # untimed oracle calls before any timed ones (steady state)
REF_STEP_S = 0.25     # length of one reference-arm step (repeated oracle calls)


def time_oracle(W: int, n_sample: int, calls: int | None, budget_s: float, threads: int,
                seed: int = 1, dist: str = "normal", warm_s: float = ORACLE_WARM_S) -> dict:
    """Times the oracle over ``n_sample`` elements drawn like the workload's partials,
    after ``warm_s`` seconds of untimed calls."""
    import oracle
    import synthetic_partials as sp
    x = sp.partials(W, n_sample, dist, seed)
    u = sp.to_u16_numpy(x)
    slots = list(u)
    out = oracle.reduce(slots, threads=threads)  # warm
    t_warm = time.perf_counter()
    while time.perf_counter() - t_warm < warm_s:
        oracle.reduce(slots, out=out, threads=threads)
    done = 0
    t0 = time.perf_counter()
    while True:
        oracle.reduce(slots, out=out, threads=threads)
        done += 1
        el = time.perf_counter() - t0
        if (calls is not None and done >= calls) or (calls is None and el >= budget_s):
            break
    el = time.perf_counter() - t0
    byts = (W + 1) * n_sample * 2 * done
    return dict(calls=done, seconds=el, bytes=byts, gbs=byts / el / 1e9, threads=threads)


def oracle_in_child(W: int, n: int, seconds: float, threads: int, seed: int, dist: str) -> dict:
    """time_oracle in a fresh Python process that never initialises CUDA.

    In a process whose CUDA context is up (with page-locked buffers
    allocated), the oracle's per-call thread start-up measured about twice as
    slow on the GB300 host as in a fresh process (16 threads: 2.4-2.5 against
    5.2-5.8 GB/s, the same 1-thread rate): the baseline is taken where the
    reference arm takes it, in a process of its own.
    """
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench.time_oracle(%d, %d, None, %r, %d, %d, %r)))"
            % (ROOT, W, n, float(seconds), threads, seed, dist))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=seconds * 4 + 120)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing child failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synthetic_partials as sp
    spec = sp.WORKLOADS[args.workload]
    W, n = spec["W"], spec["n"] or args.n
    threads = oracle.default_threads()
    # Each step is the oracle over the workload (a contiguous sample of its
    # elements where one call would take more than a second), repeated
    # enough times that a step lasts about REF_STEP_S: a 20-step run then
    # times seconds of steady-state calls, not a few milliseconds of them
    # (the oracle starts its threads per call, and single calls vary).
    per_elem_s = 2.0e-9 * W / max(1, threads) + 1e-10
    n_step = int(min(n, max(4096, 1.0 / per_elem_s)))
    calls = time_oracle(W, n_step, None, 0.5, threads, spec["seed"], spec["dist"])
    reps = max(1, int(round(REF_STEP_S / (calls["seconds"] / calls["calls"]))))
    time_oracle(W, n_step, args.warmup * reps, 0.0, threads, spec["seed"], spec["dist"], warm_s=0.0)
    r = time_oracle(W, n_step, args.steps * reps, 0.0, threads, spec["seed"], spec["dist"])
    value = r["gbs"]
    sample = (f"{args.steps} steps of {reps} oracle calls each, every call over "
              f"{'all' if n_step == n else f'the first {n_step} of'} {n} elements of the "
              f"{args.workload} partials (W={W}), {threads} threads, after {args.warmup} warm-up steps "
              f"and {ORACLE_WARM_S:.0f} s of untimed calls; a process without CUDA")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["seconds"] / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "io_dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "W": W, "n": n, "n_per_call": n_step, "calls_per_step": reps},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# GPU arm

def _graph_of_calls(torch, stream, fn, count):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(count):
            fn(i)
    return g


_FLUSH: dict = {}


def flush_l2(torch, stream, l2_bytes: int) -> None:
    """Evicts L2 with clean lines: reads a buffer of twice the L2 size on
    ``stream`` (a read, so no dirty lines are left to write back later)."""
    dev = torch.cuda.current_device()
    buf = _FLUSH.get(dev)
    if buf is None or buf.numel() < 2 * l2_bytes // 4:
        buf = _FLUSH[dev] = torch.ones(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        buf.amax()


def _timing_event(torch):
    """A timing event that a CUDA graph can record inside itself (an external
    event node), or None if this torch cannot make one."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def timed_graph_calls(torch, stream, fn, steps: int, warmup: int, chunk: int = GRAPH_CALLS,
                      sampler: ClockSampler | None = None) -> float:
    """Seconds for exactly ``steps`` calls of fn(i), launched from CUDA graphs on ``stream``.

    The start and end events are recorded by the graphs themselves.  The
    first graph opens with LEAD_IN untimed calls (the last of the warm-up
    calls), and the start event fires when the last of them completes; the
    end event fires when the last timed call completes, and LEAD_IN untimed
    calls follow it.  The timed region is thus exactly ``steps`` call
    completions of a running stream of calls -- each call overlaps its
    predecessor's tail (programmatic dependent launch), as in a long run --
    and neither the host's submission of the replay nor the GPU's launch of
    the graph falls inside it.  Before the
    timed replays L2 is flushed (the warm-up replays touched the same
    buffers), so a short run's calls read their inputs from DRAM like a long
    run's.  Without graph-recordable events (older torch) the events are
    recorded on the stream around the replays instead.
    """
    chunk = max(1, min(chunk, steps))
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    # Inputs, outputs and zero-filled workspaces were made on torch's default
    # stream; `stream` is a non-blocking stream, so order them before its calls.
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(1, min(warmup, 8))):   # eager warm-up (launch caches, lazy init)
            fn(i)
    torch.cuda.synchronize()
    start, end = _timing_event(torch), _timing_event(torch)
    in_graph = start is not None and end is not None
    if not in_graph:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
    side, side2 = torch.cuda.Stream(), torch.cuda.Stream()

    def capture(count, base, first, last):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if first and in_graph:
                for i in range(LEAD_IN):    # untimed: the stream of calls is running
                    fn(steps + i)
                side.wait_stream(stream)     # fires when the last lead-in call completes
                start.record(side)
            for i in range(count):
                fn(base + i)
            if last and in_graph:
                # The end event on a branch of its own, like the start event,
                # followed by untimed calls: both events are recorded while
                # the GPU is still launching calls, so any delay in recording
                # them is alike at both ends.
                side2.wait_stream(stream)    # fires when the last timed call completes
                end.record(side2)
                for i in range(LEAD_IN):
                    fn(steps + LEAD_IN + i)
            if first and in_graph:
                stream.wait_stream(side)
            if last and in_graph:
                stream.wait_stream(side2)
        return g

    segs = [chunk] * (steps // chunk) + ([steps % chunk] if steps % chunk else [])
    if len(segs) == 1:
        order = [capture(segs[0], 0, True, True)]
    else:
        g_first = capture(segs[0], 0, True, False)
        g_mid = capture(chunk, 0, False, False) if len(segs) > 2 else None
        g_last = capture(segs[-1], steps - segs[-1], False, True)
        order = [g_first] + [g_mid] * (len(segs) - 2) + [g_last]
    # CUDAGraph.replay() launches on torch's current stream: make it `stream`,
    # the stream the events are recorded on.
    with torch.cuda.stream(stream):
        # Warm-up replays (untimed): every graph once (its first launch
        # uploads it), then the full chunk until `warmup` calls have run.
        for g in dict.fromkeys(order):
            g.replay()
        for _ in range(max(0, (warmup - steps + chunk - 1) // chunk)):
            order[0].replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.mark_start()
        flush_l2(torch, stream, l2)
        # A bounded spin, off the clock, keeps the GPU busy while the host
        # submits the replays, so they run back to back.
        torch.cuda._sleep(QUEUE_AHEAD_CYCLES)
        if not in_graph:
            start.record(stream)
        for g in order:
            g.replay()
        if not in_graph:
            end.record(stream)
        torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    barrier()
    return start.elapsed_time(end) / 1e3


def run_native(args) -> None:
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)
    import deterministic_shot_all_gb300 as arx
    import synthetic_partials as sp

    spec = sp.WORKLOADS[args.workload]
    W, n = spec["W"], spec["n"] or args.n
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    bytes_call = (W + 1) * n * 2
    stream = torch.cuda.Stream(device=dev)

    # Inputs: the workload's partials, copied into R rotation sets (+ outputs).
    x, alias = sp.workload(args.workload, n=n)
    xd = x.to(dev)
    set_bytes = W * n * 2 + (0 if alias else n * 2)
    R = rotation_sets(set_bytes, l2)
    parts = torch.empty(R, W, n, dtype=torch.bfloat16, device=dev)
    parts.copy_(xd.unsqueeze(0).expand(R, W, n))
    outs = parts[:, 0] if alias else torch.empty(R, n, dtype=torch.bfloat16, device=dev)
    slot_lists = [[parts[k, r] for r in range(W)] for k in range(R)]

    def call(i):
        k = i % R
        arx.arx_reduce(slot_lists[k], outs[k], stream=stream)

    # Correctness of what is timed: one call checked bit for bit against the oracle.
    if rank == 0 and not args.no_check:
        import oracle
        want = oracle.reduce(list(sp.to_u16_numpy(x)))
        torch.cuda.synchronize()        # the copies above ran on the default stream
        with torch.cuda.stream(stream):
            call(0)
        torch.cuda.synchronize()
        got = sp.to_u16_numpy(outs[0].cpu())
        if not (got == want).all():
            raise SystemExit("bench: GPU output differs from the oracle; refusing to time it")
        parts[0].copy_(xd)

    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
    t = timed_graph_calls(torch, stream, call, args.steps, args.warmup, sampler=sampler)
    clocks = sampler.stop() if sampler else None
    t_max, total_bytes = aggregate_over_ranks(t, bytes_call * args.steps)
    value = total_bytes / t_max / 1e9
    per_call = t / args.steps

    extra = {}
    if not args.quick:
        extra["latency_floor"] = floor_point(torch, arx, dev, stream, l2, W, n, per_call)
        extra["hot_l2"] = hot_l2_point(torch, arx, stream, slot_lists, outs, W, n)
        extra["stream_launch"] = stream_launch_point(torch, arx, dev, stream, slot_lists, outs, R)
        extra["bandwidth"] = bandwidth_points(torch, arx, sp, dev, stream, l2)
        extra["sweep"] = {"workload": "w8_sweep_int values (integers in [-8, 8]) at W = 2, 4, 8",
                          "peak_GBs": measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS,
                          "points": {f"W{w}": sweep_points(torch, arx, dev, stream, l2, w, SWEEP_LOG2)
                                     for w in SWEEP_W}}
        extra["protocol"] = protocol_point(torch, arx, sp, dev, stream, l2, args.workload)
        extra["protocol_graph"] = protocol_graph_point(torch, arx, sp, dev, stream)
        link = pinned_copy_gbs(torch, dev)
        extra["protocol_host_slots"] = protocol_host_slots_point(torch, arx, sp, dev, stream, l2,
                                                                 args.workload, link)
        extra["external_writer"] = ext_point(torch, arx, sp, dev, stream, args.workload, link)
        extra["e2e"] = e2e_point(torch, arx, sp, dev, stream, args.workload, max(200, min(args.steps, 5000)),
                                 l2, link)
    if rank != 0:
        return
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_note = "of measured" if peak else "of fallback"
    peak = float(peak) if peak else FALLBACK_HBM_GBS
    achieved = gbs(bytes_call, per_call)
    traffic = stored_traffic(args.workload, n)
    cpu = cpu1 = None
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        r = oracle_in_child(W, n, args.cpu_seconds, threads, spec["seed"], spec["dist"])
        cpu = {"value": r["gbs"], "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{r['calls']} full calls of the {args.workload} workload "
                         f"(W={W}, n={n}) in {r['seconds']:.1f} s on {threads} host threads, after "
                         f"{ORACLE_WARM_S:.0f} s of untimed calls, in a child process without CUDA"}
        r1 = oracle_in_child(W, n, args.cpu_seconds / 2, 1, spec["seed"], spec["dist"])
        cpu1 = {"value": r1["gbs"], "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{r1['calls']} full calls in {r1['seconds']:.1f} s on 1 host thread, "
                          f"in a child process without CUDA"}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3,
        "us_per_call": per_call * 1e6, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "W": W, "n": n, "shape": [32, 4096] if n == 32 * 4096 else [n],
                   "out_aliases_slot0": alias, "l2": f"inputs rotate over {R} buffer sets "
                   f"({R * set_bytes / 1e6:.0f} MB > {ROTATE_FACTOR}x L2 {l2 / 1e6:.0f} MB); "
                   f"L2 flushed (a read of 2x its size) before the timed replay",
                   "launch": f"CUDA graphs of up to {GRAPH_CALLS} arx_reduce calls, replayed; the first "
                             f"graph opens with {LEAD_IN} untimed calls and the last closes with "
                             f"{LEAD_IN}; start and end events recorded by the graphs when the last "
                             f"untimed call before and the last timed call complete",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_note, "traffic": traffic,
                     "kernel": reduce_kernel_name(W, n, alias, props.multi_processor_count), "algorithmic_bytes_per_launch": bytes_call},
        "cpu_baseline": cpu,
        "cpu_baseline_1thread": cpu1,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


HALF_MAX_ELEMS = 1 << 22   # the library's switch from 8-byte to 16-byte vectors


def reduce_kernel_name(W: int, n: int, alias: bool, sms: int = 152) -> str:
    """The kernel the library launches for this shape (its launch policy,
    restated), with its template arguments as ncu prints them (bools as 0/1).

    Exact for the one-vector 8-byte form (128 threads per block while
    256-thread blocks would number fewer than the SMs, as at the decode-sized
    workloads; 256 for W = 5-7, or while one pass of a grid of sms x 8 blocks
    covers the n / 4 vectors with 1/16 slack), for W = 8 past that pass (the
    pipelined 16-byte form) and for the 16-byte form above 2^22 elements;
    W <= 4 messages between take a batched 8-byte form or the 16-byte one by
    the library's one-pass rule.
    """
    a = int(alias)
    if n <= HALF_MAX_ELEMS:
        blocks256 = -(-(2 * (n // 8)) // 256)
        if blocks256 < sms:
            return f"reduce_half_kernel<{W}, 128, 1, {a}>"
        if 5 <= W <= 7 or blocks256 * 16 <= sms * 8 * 17:
            return f"reduce_half_kernel<{W}, 256, 1, {a}>"
        if W == 8:
            return f"reduce_vec_kernel<8, 256, 1, 1, {a}>"
        return f"reduce_half_kernel<{W}, 256, U, {a}> (batched) or reduce_vec_kernel (one-pass rule)"
    if W <= 2:
        return f"reduce_vec_kernel<{W}, 128, 2, 1, {a}>"
    return f"reduce_vec_kernel<{W}, 256, 1, 1, {a}>"


def bandwidth_points(torch, arx, sp, dev, stream, l2) -> list:
    """GB/s at bandwidth-bound sizes, same timing method (rotation > 3x L2, graphs)."""
    pts = []
    peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
    for name, W, n, alias in (("w4_1024x8192_alias", 4, 1024 * 8192, True),
                              ("w8_sweep_int", 8, 1 << 23, False),
                              ("w8_sweep_int", 8, 1 << 27, False)):
        set_bytes = W * n * 2 + (0 if alias else n * 2)
        R = rotation_sets(set_bytes, l2, cap=64)
        # Timing only (parity at these sizes is in the tests): values drawn on the
        # device with the workload's distribution, to keep host time short.
        gen = torch.Generator(device=dev).manual_seed(3)
        if name == "w8_sweep_int":
            parts = torch.randint(-8, 9, (R, W, n), generator=gen, device=dev).to(torch.bfloat16)
        else:
            parts = (torch.randn((R, W, n), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        outs = parts[:, 0] if alias else torch.empty(R, n, dtype=torch.bfloat16, device=dev)
        slot_lists = [[parts[k, r] for r in range(W)] for k in range(R)]
        calls = 200 if n <= (1 << 23) else 40

        def call(i, slot_lists=slot_lists, outs=outs, R=R):
            arx.arx_reduce(slot_lists[i % R], outs[i % R], stream=stream)

        t = timed_graph_calls(torch, stream, call, calls, 5, chunk=calls)
        b = (W + 1) * n * 2
        g = gbs(b, t / calls)
        pts.append({"workload": name, "W": W, "n": n, "partial_MiB": n * 2 / 2**20, "in_place": alias,
                    "us_per_call": t / calls * 1e6, "GBs": g, "frac": g / peak, "rotation_sets": R})
        del parts, outs, slot_lists
        torch.cuda.empty_cache()
    return pts


def floor_point(torch, arx, dev, stream, l2, W, n, per_call) -> dict:
    """Per-call floor: the same call shape with 1 KiB partials (launch + one DRAM round trip).

    The headline message is latency-bound; its time above this floor is what
    its bytes cost, so bytes / (t - floor) is the marginal bandwidth.
    """
    n0 = 512
    R = rotation_sets((W + 1) * n0 * 2, l2, cap=4096)
    parts = torch.zeros(R, W, n0, dtype=torch.bfloat16, device=dev)
    outs = torch.empty(R, n0, dtype=torch.bfloat16, device=dev)
    lists = [[parts[k, r] for r in range(W)] for k in range(R)]

    def call(i):
        arx.arx_reduce(lists[i % R], outs[i % R], stream=stream)

    calls = 20000
    t = timed_graph_calls(torch, stream, call, calls, 100)
    floor = t / calls
    above = per_call - floor
    return {"n": n0, "us_per_call": floor * 1e6, "headline_us_above_floor": above * 1e6,
            "marginal_GBs": gbs((W + 1) * n * 2, above) if above > 0 else None}


SYNC_MODES = ("semaphore", "pad", "pad_fenced", "cluster", "semaphore_global")   # index = ARX_SYNC_*


def protocol_point(torch, arx, sp, dev, stream, l2, workload, steps: int = 2000) -> dict:
    """arx_step per step (W=8, [32,4096]) in captured graphs, fresh input sets rotating,
    for each barrier variant (Semaphore barriers with the flags in the cluster's shared
    memory; pad barrier Patterns 0/1/2; all acq_rel; the thread-block cluster barrier;
    Semaphore barriers with the flags in global memory)."""
    W, n = 8, sp.N_32x4096
    x, _ = sp.workload(workload)
    R = rotation_sets(W * n * 2 * 2, l2)
    parts = torch.empty(R, W, n, dtype=torch.bfloat16, device=dev)
    parts.copy_(x.to(dev).unsqueeze(0).expand(R, W, n))
    outs = torch.empty(R, n, dtype=torch.bfloat16, device=dev)
    lists = [[parts[k, r] for r in range(W)] for k in range(R)]
    res = {"W": W, "n": n, "steps": steps, "modes": {}}
    for mode_index, mode in enumerate(SYNC_MODES):
        ws = torch.zeros(arx.arx_ctx_workspace_bytes(W, n), dtype=torch.uint8, device=dev)
        ctx = arx.arx_ctx_init(ws, W, n)
        arx.arx_ctx_set_sync(ctx, mode_index)

        def call(i, ctx=ctx):
            arx.arx_step(ctx, lists[i % R], outs[i % R], stream=stream)

        t = timed_graph_calls(torch, stream, call, steps, 10)
        st, seq, err = arx.arx_ctx_query(ctx, stream=stream)
        res["blocks_per_rank"] = ctx.nblocks
        res["modes"][mode] = {"us_per_step": t / steps * 1e6, "status": arx.arx_status_string(st),
                              "seq": seq, "reduce_model_GBs": gbs((W + 1) * n * 2, t / steps)}
    res["us_per_step"] = res["modes"]["semaphore"]["us_per_step"]
    del parts, outs, lists
    torch.cuda.empty_cache()

    # A bandwidth-bound step: W = 8 partials of 16 MiB (n = 2^23), each
    # variant.  Traffic model per step: staging reads and writes W*n*2 bytes
    # each, the reduce reads W*n*2 and writes n*2.
    nl = 1 << 23
    Rl = rotation_sets(W * nl * 2 * 2, l2, cap=64)
    gen = torch.Generator(device=dev).manual_seed(4)
    pl = (torch.randn((Rl, W, nl), generator=gen, device=dev)).to(torch.bfloat16)
    ol = torch.empty(Rl, nl, dtype=torch.bfloat16, device=dev)
    ll = [[pl[k, r] for r in range(W)] for k in range(Rl)]
    large = {"n": nl, "modes": {}}
    model_bytes = (3 * W + 1) * nl * 2
    for mode_index, mode in enumerate(SYNC_MODES):
        ws = torch.zeros(arx.arx_ctx_workspace_bytes(W, nl), dtype=torch.uint8, device=dev)
        ctx = arx.arx_ctx_init(ws, W, nl)
        arx.arx_ctx_set_sync(ctx, mode_index)

        def call(i, ctx=ctx):
            arx.arx_step(ctx, ll[i % Rl], ol[i % Rl], stream=stream)

        t = timed_graph_calls(torch, stream, call, 200, 10, chunk=200) / 200
        st, seq, err = arx.arx_ctx_query(ctx, stream=stream)
        large["blocks_per_rank"] = ctx.nblocks
        large["modes"][mode] = {"us_per_step": t * 1e6, "status": arx.arx_status_string(st),
                                "seq": seq, "dev_err": err, "model_GBs": gbs(model_bytes, t)}
        del ws
    large["traffic_model"] = "staging 2*W*n*2 B + reduce (W+1)*n*2 B per step"
    res["large"] = large
    del pl, ol, ll
    torch.cuda.empty_cache()
    return res


def protocol_graph_point(torch, arx, sp, dev, stream) -> dict:
    """The graph workload as specified: W = 8 bf16 [32, 4096], GRAPH_STEPS (10,000)
    arx_step calls captured in ONE CUDA graph, fresh normal(0, 1) partials for
    every step (a [10000][8][n] device array, 21 GB, far beyond L2), one output
    per step.  The partials are drawn on the device here (timing only; the
    tests check every step bit for bit with the CPU-drawn seeds 4 + step).
    µs/step = graph replay time / steps; the default barrier variant, and the
    thread-block cluster barrier under "cluster"."""
    W, n, steps = 8, sp.N_32x4096, sp.GRAPH_STEPS
    inputs = torch.empty(steps, W, n, dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device=dev).manual_seed(4)
    for lo in range(0, steps, 1000):
        hi = min(steps, lo + 1000)
        inputs[lo:hi] = torch.randn((hi - lo, W, n), generator=gen, device=dev).to(torch.bfloat16)
    outputs = torch.empty(steps, n, dtype=torch.bfloat16, device=dev)
    lists = [[inputs[t, r] for r in range(W)] for t in range(steps)]
    res = None
    # The default barrier variant, then the same graph workload on the
    # thread-block cluster barrier (reported as "cluster").
    for sync in (arx.ARX_SYNC_SEMAPHORE, arx.ARX_SYNC_CLUSTER):
        ws = torch.zeros(arx.arx_ctx_workspace_bytes(W, n), dtype=torch.uint8, device=dev)
        ctx = arx.arx_ctx_init(ws, W, n)
        arx.arx_ctx_set_sync(ctx, sync)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        t0 = time.perf_counter()
        with torch.cuda.graph(g, stream=stream):
            for t in range(steps):
                arx.arx_step(ctx, lists[t], outputs[t], stream=stream)
        capture_s = time.perf_counter() - t0
        times = []
        with torch.cuda.stream(stream):
            g.replay()                      # warm-up replay (untimed)
            torch.cuda.synchronize()
            for _ in range(3):
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(QUEUE_AHEAD_CYCLES)   # replay queued when s fires
                s.record(stream)
                g.replay()
                e.record(stream)
                torch.cuda.synchronize()
                times.append(s.elapsed_time(e) / 1e3)
        st, seq, err = arx.arx_ctx_query(ctx, stream=stream)
        t = statistics.median(times)
        point = {"W": W, "n": n, "steps_per_graph": steps, "replays": len(times), "us_per_step": t / steps * 1e6,
                 "graph_ms": t * 1e3, "capture_s": capture_s, "status": arx.arx_status_string(st),
                 "seq": seq, "blocks_per_rank": ctx.nblocks}
        if res is None:
            res = point
        else:
            res["cluster"] = {k: point[k] for k in ("us_per_step", "graph_ms", "status", "seq")}
        del g, ws
    del inputs, outputs, lists
    torch.cuda.empty_cache()
    return res


def protocol_host_slots_point(torch, arx, sp, dev, stream, l2, workload, link, steps: int = 2000) -> dict:
    """arx_step with the slot banks in page-locked host memory (arx_ctx_init_split):
    every step writes the W staged partials to host memory and reads them back
    over NVLink-C2C.  Link roofline: the time the measured rate of pinned
    copies in both directions at once needs to move those bytes out and back
    (and, for reference, the one-way rates one after the other)."""
    W, n = 8, sp.N_32x4096
    x, _ = sp.workload(workload)
    R = rotation_sets(W * n * 2 * 2, l2)
    parts = torch.empty(R, W, n, dtype=torch.bfloat16, device=dev)
    parts.copy_(x.to(dev).unsqueeze(0).expand(R, W, n))
    outs = torch.empty(R, n, dtype=torch.bfloat16, device=dev)
    lists = [[parts[k, r] for r in range(W)] for k in range(R)]
    words = torch.zeros(arx.arx_ctx_words_bytes(W), dtype=torch.uint8, device=dev)
    slots = torch.empty(arx.arx_ctx_slots_bytes(W, n), dtype=torch.uint8).pin_memory()
    ctx = arx.arx_ctx_init_split(words, slots, W, n)

    def call(i):
        arx.arx_step(ctx, lists[i % R], outs[i % R], stream=stream)

    t = timed_graph_calls(torch, stream, call, steps, 10) / steps
    st, seq, err = arx.arx_ctx_query(ctx, stream=stream)
    moved = W * n * 2
    t_serial = moved / (link["d2h"] * 1e9) + moved / (link["h2d"] * 1e9)
    t_duplex = 2 * moved / (link["both"] * 1e9)
    # The same step on the thread-block cluster barrier (no Semaphore words,
    # no fault knob): the fastest host-slot form.
    words_c = torch.zeros(arx.arx_ctx_words_bytes(W), dtype=torch.uint8, device=dev)
    slots_c = torch.empty(arx.arx_ctx_slots_bytes(W, n), dtype=torch.uint8).pin_memory()
    ctx_c = arx.arx_ctx_init_split(words_c, slots_c, W, n)
    arx.arx_ctx_set_sync(ctx_c, arx.ARX_SYNC_CLUSTER)

    def call_c(i):
        arx.arx_step(ctx_c, lists[i % R], outs[i % R], stream=stream)

    tc = timed_graph_calls(torch, stream, call_c, steps, 10) / steps
    stc, seqc, _ = arx.arx_ctx_query(ctx_c, stream=stream)
    return {"W": W, "n": n, "steps": steps, "blocks_per_rank": ctx.nblocks, "us_per_step": t * 1e6,
            "status": arx.arx_status_string(st), "seq": seq,
            "link_bytes_per_step": 2 * moved,
            "roofline": {"bound": "c2c", "link_bound_us": t_duplex * 1e6, "frac": t_duplex / t,
                         "basis": "staged bytes out and back at the measured rate of pinned copies in "
                                  "both directions at once (the steps stage in turn, so writes and "
                                  "reads overlap)",
                         "serial_bound_us": t_serial * 1e6, "serial_frac": t_serial / t},
            "cluster": {"us_per_step": tc * 1e6, "frac": t_duplex / tc, "status": arx.arx_status_string(stc),
                        "seq": seqc}}


def ext_point(torch, arx, sp, dev, stream, workload, link, steps: int = 1000, warm: int = 20) -> dict:
    """The external-writer form: a host thread (standing in for arx.cu's proxy
    and NIC) raises the W flags of every step, the GPU waits for them and
    reduces the W page-locked slots over NVLink-C2C.  The slots of both banks
    hold the workload's partials, written once in place (arx_ext_slot), so the
    producer only publishes (arx_ext_publish_all, which first waits for the
    bank to be free); this times the GPU side of the hand-off.  ``steps``
    steps in one CUDA graph, the events recorded by the graph.  Link
    roofline: W*n*2 bytes read over the link per step at the measured pinned
    host->device copy rate."""
    import ctypes
    import threading
    W, n = 8, sp.N_32x4096
    x, _ = sp.workload(workload)
    words = torch.zeros(arx.arx_ext_words_bytes(), dtype=torch.uint8, device=dev)
    region = torch.zeros(arx.arx_ext_region_bytes(W, n), dtype=torch.uint8).pin_memory()
    xe = arx.arx_ext_init(words, region, W, n)
    arx.arx_ext_set_timeout(xe, 50_000_000)   # a stalled producer costs 50 ms per step, not 1 s
    for par in (0, 1):
        for r in range(W):
            ctypes.memmove(arx.arx_ext_slot(xe, par, r), x[r].data_ptr(), n * 2)
    out = torch.empty(steps, n, dtype=torch.bfloat16, device=dev)
    errors = []

    def producer(total):
        try:
            for s_ in range(1, total + 1):
                arx.arx_ext_publish_all(xe, s_, wait_s=20.0)
        except Exception as e:  # reported below
            errors.append(repr(e))

    start, end = _timing_event(torch), _timing_event(torch)
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        side.wait_stream(stream)
        start.record(side)
        for i in range(steps):
            arx.arx_ext_step(xe, out[i], stream=stream)
        end.record(stream)
        stream.wait_stream(side)
    th = threading.Thread(target=producer, args=(warm + 2 * steps,))
    th.start()
    with torch.cuda.stream(stream):
        for i in range(warm):
            arx.arx_ext_step(xe, out[i], stream=stream)
        g.replay()                      # warm-up replay (uploads the graph)
        torch.cuda.synchronize()
        torch.cuda._sleep(QUEUE_AHEAD_CYCLES)
        g.replay()
        torch.cuda.synchronize()
    th.join()
    t = start.elapsed_time(end) / 1e3 / steps
    st, seq, err = arx.arx_ext_query(xe, stream=stream)
    import oracle
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    ok = bool((sp.to_u16_numpy(out[steps - 1].cpu()) == want).all())
    moved = W * n * 2
    peak = link["h2d"]
    return {"W": W, "n": n, "steps": steps, "blocks": xe.nblocks, "us_per_step": t * 1e6,
            "status": arx.arx_status_string(st), "seq": seq, "dev_err": err, "producer_errors": errors,
            "bit_exact": ok, "metric_GBs": gbs((W + 1) * n * 2, t),
            "roofline": {"bound": "c2c", "achieved": gbs(moved, t), "peak": peak, "unit": "GB/s",
                         "frac": gbs(moved, t) / peak,
                         "basis": "W*n*2 bytes of slots read over the link per step, against the measured "
                                  "pinned host->device copy rate"}}


def pinned_copy_gbs(torch, dev, nbytes: int = 1 << 26, reps: int = 5) -> dict:
    """Best-of-reps copy-engine bandwidth between pinned host memory and the device
    (the CPU-GPU link's measured rate, the denominator of the host-buffer path)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name in ("h2d", "d2h"):
        best = float("inf")
        for _ in range(reps):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            if name == "h2d":
                d.copy_(h, non_blocking=True)
            else:
                h.copy_(d, non_blocking=True)
            e.record()
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e) / 1e3)
        out[name] = nbytes / best / 1e9
    # Both directions at once (two streams, one copy each way): the link's
    # full-duplex rate, total bytes over the time both take.
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(s1)
        s2.wait_event(s)
        with torch.cuda.stream(s1):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
        s1.wait_stream(s2)
        e.record(s1)
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    out["both"] = 2 * nbytes / best / 1e9
    out["bytes"] = nbytes
    return out


def stream_launch_point(torch, arx, dev, stream, slot_lists, outs, R) -> dict:
    """The headline call launched eagerly through the Python binding (no graph).

    back_to_back: K calls enqueued in a row, events around the batch (bound by the
    host's launch rate); single_call: events around one call at a time, GPU idle
    before each, median over the calls (includes the launch latency); the plan_
    figures: the same through a prepared arx_reduce_plan (one C call per call).
    """
    def call(i):
        arx.arx_reduce(slot_lists[i % R], outs[i % R], stream=stream)

    K = 2000
    with torch.cuda.stream(stream):
        for i in range(50):
            call(i)
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for i in range(K):
            call(i)
        e.record(stream)
        torch.cuda.synchronize()
        b2b = s.elapsed_time(e) / 1e3 / K
        single = []
        for i in range(1000):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            call(i)
            e.record(stream)
            e.synchronize()
            single.append(s.elapsed_time(e) / 1e3)
        # The same calls through prepared plans (arguments marshalled once).
        plans = [arx.arx_reduce_plan(slot_lists[k], outs[k], stream=stream) for k in range(R)]
        for i in range(50):
            plans[i % R]()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for i in range(K):
            plans[i % R]()
        e.record(stream)
        torch.cuda.synchronize()
        b2b_plan = s.elapsed_time(e) / 1e3 / K
        single_plan = []
        for i in range(1000):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            plans[i % R]()
            e.record(stream)
            e.synchronize()
            single_plan.append(s.elapsed_time(e) / 1e3)
    return {"back_to_back_us_per_call": b2b * 1e6, "calls": K,
            "single_call_us_median": statistics.median(single) * 1e6, "single_calls": len(single),
            "plan_back_to_back_us_per_call": b2b_plan * 1e6,
            "plan_single_call_us_median": statistics.median(single_plan) * 1e6}


def hot_l2_point(torch, arx, stream, slot_lists, outs, W, n) -> dict:
    """HOT-L2 figure, labelled as such: the same buffer set every call, so the
    inputs are served from L2 (not the headline, which rotates beyond L2)."""
    def call(i):
        arx.arx_reduce(slot_lists[0], outs[0], stream=stream)

    calls = 20000
    t = timed_graph_calls(torch, stream, call, calls, 100)
    return {"label": "hot L2 (one buffer set reused)", "us_per_call": t / calls * 1e6,
            "GBs": gbs((W + 1) * n * 2, t / calls)}


def e2e_point(torch, arx, sp, dev, stream, workload, steps, l2, link) -> dict:
    """The metric through arx_reduce_host: pinned host partials in, host result out, per step.

    The host sets rotate like the device ones (footprint above 3x L2): the GPU
    caches host memory it reads over the CPU-GPU link, so one set would hit.
    """
    x, _ = sp.workload(workload)
    W, n = x.shape
    R = rotation_sets((W + 1) * n * 2, l2)
    host = torch.empty(R, W, n, dtype=torch.bfloat16).pin_memory()
    host.copy_(x.unsqueeze(0).expand(R, W, n))
    hout = torch.empty(R, n, dtype=torch.bfloat16).pin_memory()
    lists = [[host[k, r] for r in range(W)] for k in range(R)]
    staging = torch.empty(arx.arx_reduce_host_staging_bytes(W, n), dtype=torch.uint8, device=dev)

    def call(i):
        arx.arx_reduce_host(lists[i % R], hout[i % R], staging, stream=stream)

    t = timed_graph_calls(torch, stream, call, steps, 5, chunk=min(steps, 1000))
    import oracle
    want = oracle.reduce(list(sp.to_u16_numpy(x)))
    ok = bool((sp.to_u16_numpy(hout[(steps - 1) % R]) == want).all())
    value = gbs((W + 1) * n * 2, t / steps)

    # For comparison, the conventional form of the same end-to-end call: the
    # partials copied in from the same page-locked buffers by the copy engine,
    # arx_reduce on the device, the sum copied back.
    dparts = torch.empty(W, n, dtype=torch.bfloat16, device=dev)
    dout = torch.empty(n, dtype=torch.bfloat16, device=dev)
    dlist = [dparts[r] for r in range(W)]

    def staged(i):
        k = i % R
        dparts.copy_(host[k], non_blocking=True)
        arx.arx_reduce(dlist, dout, stream=stream)
        hout[k].copy_(dout, non_blocking=True)

    t2 = timed_graph_calls(torch, stream, staged, steps, 5, chunk=min(steps, 1000))
    ok2 = bool((sp.to_u16_numpy(hout[(steps - 1) % R]) == want).all())
    # Link roofline: the W partials cross the CPU-GPU link host-to-device and
    # the sum device-to-host, the two directions at once; the bound is the
    # slower direction's bytes at the measured pinned copy rate (here the
    # partials', host-to-device).
    t_call = t / steps
    h2d_s = W * n * 2 / (link["h2d"] * 1e9)
    d2h_s = n * 2 / (link["d2h"] * 1e9)
    bound_s = max(h2d_s, d2h_s)
    peak = link["h2d"] if h2d_s >= d2h_s else link["d2h"]
    return {"value": value, "unit": "GB/s",
            "us_per_call": t_call * 1e6, "steps": steps,
            "h2d_bytes_per_step": W * n * 2, "d2h_bytes_per_step": n * 2, "bit_exact": ok,
            "roofline": {"bound": "c2c", "achieved": (W * n * 2 if h2d_s >= d2h_s else n * 2) / t_call / 1e9,
                         "peak": peak, "unit": "GB/s", "frac": bound_s / t_call,
                         "link_bound_us": bound_s * 1e6,
                         "basis": "the binding direction's bytes per call (the W partials, host to device; "
                                  "the sum crosses the other way at the same time) at the measured pinned "
                                  "copy rate",
                         "peak_source": f"measured in this run: pinned host->device copy of "
                                        f"{link['bytes'] >> 20} MiB (device->host {link['d2h']:.0f} GB/s)"},
            "path": "arx_reduce_host on page-locked host buffers: the kernel reads the partials "
                    "and writes the sum in host memory over NVLink-C2C (no staging copies); "
                    f"{R} rotating host sets",
            "copy_engine_form": {"us_per_call": t2 / steps * 1e6, "GBs": gbs((W + 1) * n * 2, t2 / steps),
                                 "bit_exact": ok2,
                                 "path": "pinned partials copied in by the copy engine, arx_reduce, "
                                         "sum copied back, same buffers and graphs"}}


def sweep_points(torch, arx, dev, stream, l2, W: int, log2_sizes) -> list:
    """GB/s of arx_reduce against size for the integer sweep workload (W partials
    of 2^k elements, k in ``log2_sizes``), by the headline's method (graph
    replays, rotation footprint above 3x L2, L2 flushed before the timed
    calls).  Values are drawn on the device (timing only; parity at every size
    is in the tests)."""
    peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
    pts = []
    for k in log2_sizes:
        n = 1 << k
        set_bytes = (W + 1) * n * 2
        R = rotation_sets(set_bytes, l2)
        gen = torch.Generator(device=dev).manual_seed(3)
        parts = torch.randint(-8, 9, (R, W, n), generator=gen, device=dev).to(torch.bfloat16)
        outs = torch.empty(R, n, dtype=torch.bfloat16, device=dev)
        lists = [[parts[j, r] for r in range(W)] for j in range(R)]

        def call(i, lists=lists, outs=outs, R=R):
            arx.arx_reduce(lists[i % R], outs[i % R], stream=stream)

        calls = int(min(20000, max(20, 2e9 // set_bytes)))
        t = timed_graph_calls(torch, stream, call, calls, 20, chunk=min(calls, GRAPH_CALLS))
        g = gbs(set_bytes, t / calls)
        pts.append({"log2_n": k, "n": n, "partial_bytes": 2 * n, "calls": calls,
                    "us_per_call": t / calls * 1e6, "GBs": g, "frac": g / peak})
        del parts, outs, lists
        torch.cuda.empty_cache()
    return pts


SWEEP_W = (2, 4, 8)
SWEEP_LOG2 = (19, 20, 21, 22, 23)     # 1 MiB .. 16 MiB per partial


def run_sweep(args) -> None:
    """GB/s vs per-partial size for the integer sweep workload (W = --sweep-w,
    n = 2^--sweep-min .. 2^--sweep-max); prints one JSON object."""
    import torch
    import deterministic_shot_all_gb300 as arx
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    stream = torch.cuda.Stream(device=dev)
    peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
    pts = sweep_points(torch, arx, dev, stream, l2, args.sweep_w, range(args.sweep_min, args.sweep_max + 1))
    print(json.dumps({"sweep": "arx_reduce", "W": args.sweep_w, "peak_GBs": peak,
                      "peak_source": "of measured" if measured_peaks().get("hbm_gbs") else "of fallback",
                      "points": pts}), flush=True)


def run_protocol(args) -> None:
    """Only the protocol step (W = 8 bf16 [32, 4096], every barrier variant, --steps
    steps each in graphs); prints one JSON object.  Used to profile the step kernel."""
    import torch
    import deterministic_shot_all_gb300 as arx
    import synthetic_partials as sp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2**20)
    stream = torch.cuda.Stream(device=dev)
    res = protocol_point(torch, arx, sp, dev, stream, l2, DEFAULT_WORKLOAD, steps=args.steps)
    print(json.dumps({"protocol": res}), flush=True)


def run_protocol_host(args) -> None:
    """Only the protocol step with its slot banks in page-locked host memory
    (W = 8 bf16 [32, 4096], --steps steps in graphs); prints one JSON object.
    Used to profile the staggered host-slot step."""
    import torch
    import deterministic_shot_all_gb300 as arx
    import synthetic_partials as sp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2**20)
    stream = torch.cuda.Stream(device=dev)
    link = pinned_copy_gbs(torch, dev)
    res = protocol_host_slots_point(torch, arx, sp, dev, stream, l2, DEFAULT_WORKLOAD, link, steps=args.steps)
    print(json.dumps({"protocol_host_slots": res, "link": link}), flush=True)


def run_ext(args) -> None:
    """Only the external-writer step (W = 8 bf16 [32, 4096], --steps steps in one
    graph); prints one JSON object.  Used to profile its kernel."""
    import torch
    import deterministic_shot_all_gb300 as arx
    import synthetic_partials as sp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    link = pinned_copy_gbs(torch, dev)
    res = ext_point(torch, arx, sp, dev, stream, DEFAULT_WORKLOAD, link, steps=args.steps)
    print(json.dumps({"external_writer": res, "link": link}), flush=True)


def main(argv=None) -> None:
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200000)
    p.add_argument("--warmup", type=int, default=1000)
    p.add_argument("--impl", choices=("native", "reference"), default="native")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=["w2_32x4096_uniform", "w8_32x4096_normal", "w4_1024x8192_alias", "w8_sweep_int"])
    p.add_argument("--n", type=int, default=1 << 23, help="elements per partial for w8_sweep_int")
    p.add_argument("--quick", action="store_true", help="headline only (no bandwidth/protocol/e2e)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-check", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--sweep", action="store_true", help="GB/s vs size curve instead of the headline")
    p.add_argument("--sweep-w", type=int, default=8)
    p.add_argument("--sweep-min", type=int, default=9)
    p.add_argument("--sweep-max", type=int, default=27)
    p.add_argument("--protocol", action="store_true", help="only the protocol step, every barrier variant")
    p.add_argument("--protocol-host", action="store_true",
                   help="only the protocol step with its slots in page-locked host memory")
    p.add_argument("--ext", action="store_true",
                   help="only the external-writer step (host producer, GPU consumer)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.steps < 1:
        p.error("--steps must be >= 1")
    if args.sweep:
        run_sweep(args)
    elif args.protocol:
        run_protocol(args)
    elif args.protocol_host:
        run_protocol_host(args)
    elif args.ext:
        run_ext(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
