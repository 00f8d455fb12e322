"""Benchmark of the layer-wise paged KV block reshuffle on one GB300 (or N replicas).

One step = the whole hot path over one batch: the batch plan, then for every layer
slice (hit_layer[l]), merge-scatter (hit + miss into the paged pool), gather (pool ->
per-layer K/V objects) and scatter-back (objects -> pool).  The ops run phase by
phase (all layers of one op, then the next op), so no kernel finds its inputs in L2:
every phase streams at least 8 GB through a 129 MB L2.

Prints one JSON line.  `value` is algorithmic bytes moved (read + write, every op)
per second of the timed region, in GB/s; `roofline` is the dominant kernel's
achieved bandwidth against the measured HBM copy peak; `e2e` repeats the step with
the inputs copied from pinned host memory and the objects read back inside the timed
region; `cpu_baseline` is the CPU oracle on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference   # the CPU oracle on the host cores
"""
from __future__ import annotations

import argparse
import copy
import dataclasses
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "KV reshuffle HBM GB/s (read+write) and % of GB300 peak; µs per layer"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "llama3_8b_agentic"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, vendor figure (context for "% of peak")
HIT_RING = 8
KERNEL_REPS = 11  # replays whose per-phase events give the per-kernel median
OPS = ("slice", "merge_scatter", "gather", "scatter_back")
KERNEL_NAMES = {"slice": "kvl_slice_kernel", "merge_scatter": "kvl_merge_scatter_kernel",
                "gather": "kvl_gather_kernel", "scatter_back": "kvl_scatter_back_kernel"}


# ---------------------------------------------------------------------------
# Bytes each op moves (algorithmic: each byte read once and written once)
# ---------------------------------------------------------------------------

def op_bytes(spec) -> dict:
    """Algorithmic read+write bytes of one launch of each op (one layer, whole batch)."""
    R = spec.R
    hit = int(sum(spec.t_hit))
    tokens = int(spec.t_all().sum())
    blocks = int(spec.nblk().sum())
    return {"slice": 2 * hit * R, "merge_scatter": 2 * tokens * R,
            "gather": 2 * spec.P * blocks * spec.B * spec.Rp,
            "scatter_back": 2 * spec.P * blocks * spec.B * spec.Rp}


def step_bytes(spec) -> int:
    return spec.L * sum(op_bytes(spec).values())


def describe(spec) -> dict:
    d = dict(workload=spec.name, L=spec.L, P=spec.P, B=spec.B, Rp=spec.Rp,
             requests=spec.n_req, T_hit=int(sum(spec.t_hit)), T_miss=int(sum(spec.t_miss)),
             pool_blocks=spec.n_pool, payload={"normal": "bf16 N(0,1)",
                                                "uniform2": "bf16 U[-2,2]"}.get(spec.values, spec.values),
             objects_layout={"layer": "[L][P][nblk][B][Rp]",
                             "block": "[nblk][L][P][B][Rp] (one file of 2L objects per block)"}
             [spec.objects],
             step="plan, then per layer slice, merge-scatter, gather, scatter-back "
                  "(each op over all layers before the next op)",
             l2="inputs larger than L2: every phase streams >= 8 GB past a 129 MB L2")
    if spec.name == "llama3_8b_agentic":
        d.update(H_kv=8, d=128)
    return d


# ---------------------------------------------------------------------------
# Multi-rank plumbing (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int, path: Path | None):
        self.proc, self.path, self.gpu = None, path, gpu_index

    def __enter__(self):
        try:
            self.out = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out if self.path else subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            self.text = ""
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        if self.path:
            self.out.close()
            out = self.path.read_text()
        self.text = out or ""
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.text.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Peaks and ncu traffic records
# ---------------------------------------------------------------------------

def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        v = float(json.loads(p.read_text())["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the code the kernels are built from (the CUDA sources and the C ABI
    header), comments and blank lines left out, so that a change of wording does not
    make a recorded ncu measurement stale."""
    h = hashlib.sha256()
    files = sorted((ROOT / "layer_wise_paged_gb300" / "csrc").glob("*")) + [ROOT / "include" / "kvl.h"]
    for f in files:
        text = re.sub(r"/\*.*?\*/", "", f.read_text(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.strip() for line in text.splitlines() if line.strip())
        h.update(f.name.encode() + b"\0" + code.encode() + b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu record (profiles/dram_traffic.txt),
    if it was taken on this kernel source, else None."""
    p = ROOT / "profiles" / "dram_traffic.txt"
    try:
        lines = p.read_text().splitlines()
    except OSError:
        return None
    for line in lines:
        f = line.split()
        if len(f) == 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload \
                and f[2] == kernel_source_hash():
            return int(f[3])
    return None


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def phase_launch_flags(op, i, l0, *, ring, n_launches, shared_objects, serial):
    """Flags of launch i (first layer l0) of an op's phase of n_launches launches.

    A launch may overlap the one before it only when the two touch disjoint bytes:
    never the first launch of a phase (it reads the previous phase's output), never a
    slice launch that reuses a buffer of the hit_layer ring (l0 a multiple of `ring`),
    and no gather or scatter-back launch when all layers share one layer of objects.
    The launch before a run of overlapping ones leaves them half of each SM."""
    from layer_wise_paged_gb300 import KVL_LAUNCH_OVERLAP_PREVIOUS, KVL_LAUNCH_SHARE_SMS
    if serial or (shared_objects and op in ("gather", "scatter_back")):
        return 0
    if i == 0 or (op == "slice" and l0 % ring == 0):
        return KVL_LAUNCH_SHARE_SMS if n_launches > 1 else 0
    return KVL_LAUNCH_OVERLAP_PREVIOUS


def _layer_shifted(requests, layer):
    """Request layouts whose layer-0 view is `layer` of the original (pointer shift)."""
    return [dataclasses.replace(q, hit_off=q.hit_off + layer * q.hit_layer_stride,
                                miss_off=q.miss_off + layer * q.miss_layer_stride,
                                obj_layer_stride=0) for q in requests]


class OracleSample:
    """Host buffers for the CPU oracle: the workload's full inputs (shared, read only),
    a one-layer pool and one layer of objects; `run(layer)` does the step's four ops
    for that layer.  `worker()` gives another sample over the same inputs with its own
    pool and objects, so that several threads can run layers at once (the oracle's C
    calls release the GIL)."""

    def __init__(self, spec, hit=None, miss=None):
        import torch
        import oracle
        self.spec = spec
        lay = workloads.layout(spec, objects_one_layer=True)
        self.lay = lay
        if hit is None:
            t = torch.empty(lay.hit_bytes, dtype=torch.uint8)
            workloads.fill_payload(t, spec.values, spec.seed * 7 + 1)
            hit = t.numpy()
            t = torch.empty(max(16, lay.miss_bytes), dtype=torch.uint8)
            workloads.fill_payload(t, spec.values, spec.seed * 7 + 2)
            miss = t.numpy()
        self.hit, self.miss = hit, miss
        self.tables = workloads.block_tables(spec)
        self.src_tables = workloads.source_tables(spec)
        self.g1 = dataclasses.replace(spec, L=1)
        self.oracle = oracle
        self._own_buffers()

    def _own_buffers(self):
        spec = self.spec
        self.pool = np.full(spec.P * spec.n_pool * spec.B * spec.Rp, workloads.SENTINEL, np.uint8)
        self.objects = np.full(max(16, self.lay.obj_bytes), workloads.SENTINEL, np.uint8)

    def worker_bytes(self) -> int:
        """Host bytes one more worker allocates."""
        return self.pool.nbytes + self.objects.nbytes

    def worker(self) -> "OracleSample":
        w = copy.copy(self)
        w._own_buffers()
        return w

    def run(self, layer: int) -> int:
        ob = self.oracle.Batch(self.g1, _layer_shifted(self.lay.requests, layer), self.hit,
                               self.miss, self.objects, self.tables, self.src_tables)
        st, _ = ob.slice_layer(0)
        s2, _ = ob.merge_scatter(0, self.pool)
        s3 = ob.gather_objects(0, self.pool)
        s4 = ob.scatter_back(0, self.pool)
        if st or s2 or s3 or s4:
            raise RuntimeError("oracle reported an error on the benchmark workload")
        return sum(op_bytes(self.spec).values())


def host_cpu() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
    if m:
        return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
    name = {("0x41", "0xd4f"): "Arm Neoverse V2"}.get(
        (imp and imp.group(1), part and part.group(1)), "")
    return " ".join(x for x in (platform.machine(), name,
                                imp and f"implementer {imp.group(1)}",
                                part and f"part {part.group(1)}") if x)


def oracle_threads(sample, want=None) -> int:
    """Worker threads for the oracle: every host core, as far as host memory allows
    (half of what is available goes to the workers' own pools and objects)."""
    cores = os.cpu_count() or 1
    want = cores if want is None else max(1, min(int(want), cores))
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        return 1
    return max(1, min(want, int(avail // 2 // max(1, sample.worker_bytes()))))


def oracle_workers(sample, threads):
    """`threads` samples over the same inputs, each with its own pool and objects."""
    return [sample] + [sample.worker() for _ in range(threads - 1)]


def time_oracle(workers, layers, budget_s):
    """Run the oracle over `layers` (each: the step's four ops on one layer), one
    thread per worker, each taking the next layer until the list or the time budget
    (checked before each layer) runs out.  Returns (bytes, seconds, layers done)."""
    import threading
    lock, todo, done = threading.Lock(), list(layers), []
    t0 = time.perf_counter()

    def loop(w):
        while True:
            with lock:
                if not todo or (done and time.perf_counter() - t0 > budget_s):
                    return
                layer = todo.pop(0)
            n = w.run(layer)
            with lock:
                done.append(n)

    ts = [threading.Thread(target=loop, args=(w,)) for w in workers]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return sum(done), time.perf_counter() - t0, len(done)


def cpu_baseline(spec, budget_s=12.0, sample=None, threads=None):
    """The oracle on the host cores: one thread, then every core, each timed on the
    workload's layers, in order and over again, until its half of `budget_s` is spent
    (at least one layer).  The all-cores figure is the baseline's value."""
    sample = sample or OracleSample(spec)
    n = oracle_threads(sample, threads)
    workers = oracle_workers(sample, n)
    layers = [i % spec.L for i in range(spec.L * 1000)]
    b1, t1, l1 = time_oracle(workers[:1], layers, budget_s / 2)
    bn, tn, ln = time_oracle(workers, layers, budget_s / 2)
    return {"value": round(bn / tn / 1e9, 3), "unit": UNIT, "cores": n, "kind": "oracle",
            "single_thread_value": round(b1 / t1 / 1e9, 3),
            "cpu": host_cpu(), "cores_available": os.cpu_count(),
            "sample": f"{spec.name}: {ln} layer passes over its {spec.L} layers (all four "
                      f"ops each) on {n} threads, {bn / 1e9:.2f} GB algorithmic in {tn:.1f} s; "
                      f"single thread: {l1} layers, {b1 / 1e9:.2f} GB in {t1:.1f} s; plain C "
                      f"oracle, one layer per call"}


def bench_spec(args):
    """The named workload, or its first --layers layers (a smaller case of the same
    kernels, for profiling captures that must fit in a few GB)."""
    spec = workloads.get_spec(args.workload)
    if args.layers:
        spec = dataclasses.replace(spec, L=min(spec.L, args.layers))
    if args.objects != spec.objects:
        spec = dataclasses.replace(spec, objects=args.objects)
    return spec


def run_reference(args):
    """The CPU oracle as the reference arm, on every host core: each step runs the four
    ops on one layer per worker thread (successive layers of the workload)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    spec = bench_spec(args)
    sample = OracleSample(spec)
    n = oracle_threads(sample)
    workers = oracle_workers(sample, n)
    layer = 0

    def step():
        nonlocal layer
        ls = [(layer + i) % spec.L for i in range(n)]
        layer = (layer + n) % spec.L
        return time_oracle(workers, ls, float("inf"))

    for _ in range(args.warmup):
        step()
    total, dt = 0, 0.0
    for _ in range(args.steps):
        b, t, _ = step()
        total, dt = total + b, dt + t
    v = total / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": dict(describe(spec), us_per_layer=round(dt / args.steps / n * 1e6, 1),
                           layers_per_s=round(args.steps * n / dt, 3)),
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": n, "kind": "oracle",
                             "cpu": host_cpu(), "cores_available": os.cpu_count(),
                             "sample": f"{spec.name}: each step one layer (all four ops) on "
                                       f"each of {n} threads, plain C oracle"},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------

class BenchStep:
    """The buffers and launches of one bench step on a workload.

    A step is the plan, then every layer's slice, merge-scatter, gather and
    scatter-back, op by op (all layers of one op, then the next), K layers per launch.
    hit_layer[l] goes to a ring of HIT_RING per-layer buffers: each is rewritten only
    after several other layers' traffic has pushed its lines out of L2.  The largest
    workloads keep one layer of objects (object layer stride 0, each layer's gather
    lands in the same > L2-sized region) to fit in HBM."""

    def __init__(self, spec, dev, layers_per_launch=1, serial=False):
        import torch
        from layer_wise_paged_gb300.batch import Batch
        self.spec, self.serial = spec, serial
        self.one_layer = workloads.footprint_bytes(spec) > 160e9
        self.bufs = workloads.allocate(spec, dev, objects_one_layer=self.one_layer)
        lay = self.bufs["layout"]
        self.geom = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
        self.batch = Batch(self.geom, lay.requests, self.bufs["hit"], self.bufs["miss"],
                           self.bufs["objects"], self.bufs["tables"], self.bufs["src_tables"])
        self.pool = self.bufs["pool"]
        self.K = K = max(1, min(layers_per_launch, spec.L))
        self.groups = [(l0, min(K, spec.L - l0)) for l0 in range(0, spec.L, K)]
        self.ring = min(spec.L, -(-max(HIT_RING, K) // K) * K)
        self.layer_hit = self.batch.total_hit * spec.R
        self.hit_out = torch.empty(max(16, self.ring * self.layer_hit), dtype=torch.uint8,
                                   device=dev)
        self.hit_views = [self.hit_out[(l % self.ring) * self.layer_hit:] for l in range(spec.L)]

    def flags(self, op, i, l0):
        """Launch flags of launch i (first layer l0) of op's phase (phase_launch_flags)."""
        return phase_launch_flags(op, i, l0, ring=self.ring, n_launches=len(self.groups),
                                  shared_objects=self.one_layer, serial=self.serial)

    def phases(self, b, s):
        """(op, [launch thunks]) for each phase of batch b's step on stream s."""
        pool, hv = self.pool, self.hit_views
        calls = {
            "slice": lambda l, n, f: b.slice_layer(l, hv[l], s, layer_count=n, flags=f),
            "merge_scatter": lambda l, n, f: b.merge_scatter(l, pool, None, s, layer_count=n, flags=f),
            "gather": lambda l, n, f: b.gather(l, pool, s, layer_count=n, flags=f),
            "scatter_back": lambda l, n, f: b.scatter_back(l, pool, s, layer_count=n, flags=f),
        }
        return [(op, [(lambda fn=calls[op], l0=l0, n=n, f=self.flags(op, i, l0): fn(l0, n, f))
                      for i, (l0, n) in enumerate(self.groups)]) for op in OPS]

    def enqueue(self, b, s, events=None):
        """One step of batch b on stream s; events[op] = (start, end) around each phase."""
        b.plan(stream=s)
        for op, launches in self.phases(b, s):
            # one event pair per phase, around all of its launches: an event between two
            # kernels would end the programmatic dependent launch between them
            if events is not None:
                events[op][0].record(s)
            for launch in launches:
                launch()
            if events is not None:
                events[op][1].record(s)


def capture_step_graph(dev, stream, fn):
    """A CUDA graph of fn(stream): one eager run on a side stream first (outside capture,
    so the library's per-device caches are filled), then the capture."""
    import torch
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        fn(cap)
    cap.synchronize()
    with torch.cuda.graph(graph, stream=cap):
        fn(torch.cuda.current_stream(dev))
    stream.wait_stream(cap)
    return graph


def run_gpu(args):
    import torch
    import layer_wise_paged_gb300 as kvl
    from layer_wise_paged_gb300.batch import Batch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    kvl.build()
    kvl.lib()

    spec = bench_spec(args)
    bs = BenchStep(spec, dev, layers_per_launch=args.layers_per_launch,
                   serial=args.serial_launches)
    bufs, lay, g, batch = bs.bufs, bs.bufs["layout"], bs.geom, bs.batch
    K, groups, ring, one_layer = bs.K, bs.groups, bs.ring, bs.one_layer
    launch_flags = bs.flags
    stream = torch.cuda.current_stream(dev)

    def make_event():
        try:  # a record node when captured in a CUDA graph
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None

    def run_step(b, s, events):
        bs.enqueue(b, s, events)

    def step(events=None, s=None):
        run_step(batch, s or stream, events)

    launches_per_step = kvl.kvl_launches_per_call(0) + len(groups) * 4
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    code, detail = batch.status(stream)
    if code != 0:
        raise SystemExit(f"bench.py: plan status {code} detail {detail}")

    # One step captured as a CUDA graph (the launches of the C-ABI calls, with a
    # timing event recorded on the launch stream around each kernel), replayed once
    # per timed step.  --eager launches through the C ABI from Python every step.
    ev = None
    graph = None
    if not args.eager and make_event() is not None:
        ev = {op: (make_event(), make_event()) for op in OPS}
        graph = capture_step_graph(dev, stream, lambda s_: run_step(batch, s_, ev))
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
    eager_ev = {op: [] for op in OPS}

    def timed_step():
        if graph is not None:
            graph.replay()
        else:
            evs = {op: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for op in OPS}
            step(evs)
            for op in OPS:
                eager_ev[op].append(evs[op])

    clocks_path = Path(args.clocks_csv) if args.clocks_csv else None
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, clocks_path) as clk:
        time.sleep(0.3)
        t0.record(stream)
        for _ in range(args.steps):
            timed_step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    elapsed = t0.elapsed_time(t1) / 1e3
    elapsed = max_over_ranks(elapsed, dist, dev)
    code, detail = batch.status(stream)
    if code != 0:
        raise SystemExit(f"bench.py: status {code} detail {detail} after the timed steps")
    # per-launch durations: each op's phase time over its launches, the median over
    # timed steps.  Eager mode keeps every timed step's events; a graph's events hold
    # its last replay, so after the timed region the graph is replayed KERNEL_REPS more
    # times, each read back on its own (these replays are not part of `value`).
    if graph is not None:
        phase_s = {op: [] for op in OPS}
        for _ in range(KERNEL_REPS):
            graph.replay()
            torch.cuda.synchronize(dev)
            for op in OPS:
                phase_s[op].append(ev[op][0].elapsed_time(ev[op][1]) / 1e3)
        code, detail = batch.status(stream)
        if code != 0:
            raise SystemExit(f"bench.py: status {code} detail {detail} after the timing replays")
    else:
        phase_s = {op: [a.elapsed_time(b) / 1e3 for a, b in eager_ev[op]] for op in OPS}

    sb = step_bytes(spec)
    value = world * sb * args.steps / elapsed / 1e9
    per_op = {}
    for op in OPS:
        ts = [t / len(groups) for t in phase_s[op]]
        avg = statistics.median(ts)
        per_op[op] = {"us_per_launch": round(avg * 1e6, 2),
                      "gbs": round(op_bytes(spec)[op] * spec.L / len(groups) / avg / 1e9, 1),
                      "layers_per_s": round(spec.L / len(groups) / avg, 1),
                      "total_s": avg * len(groups)}
    dom = max(OPS, key=lambda o: per_op[o]["total_s"])
    peak, peak_kind = hbm_peak()
    achieved = per_op[dom]["gbs"]
    # the pipeline depth most of the dominant op's launches ran with (the kernels are
    # instantiated per depth: 3 stages when sharing SMs with a neighbour launch, else 6)
    shares = launch_flags(dom, 1, groups[1][0]) if len(groups) > 1 else 0
    kname = f"{KERNEL_NAMES[dom]}<{3 if shares else 6}>"
    traffic = recorded_traffic(kname, spec.name) if K == 1 else None
    roofline = {"bound": "hbm", "kernel": kname + f" ({dom})",
                "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "algorithmic_bytes_per_launch": op_bytes(spec)[dom] * spec.L // len(groups),
                "traffic": traffic}
    kernels = {op: {k: v for k, v in per_op[op].items() if k != "total_s"} for op in OPS}

    # ---- end to end: pinned host inputs in, objects out, inside the timed region.
    # Two sets of device inputs and objects: step s uploads into set s % 2 on one copy
    # stream and reads its objects back on another, so step s+1's upload and step
    # s-1's read-back overlap step s's kernels.  Every step still copies its own
    # inputs in and its own objects out inside the timed region.
    e2e = None
    if not args.no_e2e:
        h_hit = torch.empty(bufs["hit"].numel(), dtype=torch.uint8, pin_memory=True)
        h_miss = torch.empty(bufs["miss"].numel(), dtype=torch.uint8, pin_memory=True)
        h_tab = torch.empty(bufs["tables"].numel(), dtype=torch.int32, pin_memory=True)
        h_obj = [torch.empty(bufs["objects"].numel(), dtype=torch.uint8, pin_memory=True)
                 for _ in range(2)]
        h_hit.copy_(bufs["hit"])
        h_miss.copy_(bufs["miss"])
        h_tab.copy_(bufs["tables"])
        h_in = h_hit.numel() + h_miss.numel() + 4 * h_tab.numel()
        h_out = h_obj[0].numel()
        sets = [dict(hit=bufs["hit"], miss=bufs["miss"], tables=bufs["tables"],
                     objects=bufs["objects"], batch=batch, graph=graph)]
        second = dict(hit=torch.empty_like(bufs["hit"]), miss=torch.empty_like(bufs["miss"]),
                      tables=torch.empty_like(bufs["tables"]),
                      objects=torch.empty_like(bufs["objects"]))
        second["batch"] = Batch(g, lay.requests, second["hit"], second["miss"], second["objects"],
                                second["tables"], bufs["src_tables"])
        second["graph"] = None
        if graph is not None:
            second["graph"] = capture_step_graph(
                dev, stream, lambda s_: run_step(second["batch"], s_, None))
        sets.append(second)
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_run(n):
            h2d.wait_stream(stream)
            d2h.wait_stream(stream)
            for i in range(n):
                k = i % 2
                st = sets[k]
                if i >= 2:
                    h2d.wait_event(ev_comp[k])  # step i-2 no longer reads set k's inputs
                with torch.cuda.stream(h2d):
                    st["hit"].copy_(h_hit, non_blocking=True)
                    st["miss"].copy_(h_miss, non_blocking=True)
                    st["tables"].copy_(h_tab, non_blocking=True)
                    ev_in[k].record(h2d)
                stream.wait_event(ev_in[k])
                if i >= 2:
                    stream.wait_event(ev_out[k])  # step i-2's objects are on the host
                if st["graph"] is not None:
                    st["graph"].replay()
                else:
                    run_step(st["batch"], stream, None)
                ev_comp[k].record(stream)
                d2h.wait_event(ev_comp[k])
                with torch.cuda.stream(d2h):
                    h_obj[k].copy_(st["objects"], non_blocking=True)
                    ev_out[k].record(d2h)
            stream.wait_stream(h2d)
            stream.wait_stream(d2h)

        def link_rates():
            """The copy engines' rates on this machine for the step's own transfers: inputs
            in alone, objects out alone, and both at once (GB/s, best of 3)."""
            def timed(fn):
                best = None
                for _ in range(3):
                    torch.cuda.synchronize(dev)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    h2d.wait_stream(stream)
                    d2h.wait_stream(stream)
                    fn()
                    stream.wait_stream(h2d)
                    stream.wait_stream(d2h)
                    b.record(stream)
                    torch.cuda.synchronize(dev)
                    t = a.elapsed_time(b) / 1e3
                    best = t if best is None else min(best, t)
                return best

            def up():
                with torch.cuda.stream(h2d):
                    second["hit"].copy_(h_hit, non_blocking=True)
                    second["miss"].copy_(h_miss, non_blocking=True)
                    second["tables"].copy_(h_tab, non_blocking=True)

            def down():
                with torch.cuda.stream(d2h):
                    h_obj[1].copy_(second["objects"], non_blocking=True)

            t_up, t_down = timed(up), timed(down)
            t_both = timed(lambda: (up(), down()))
            return {"h2d_gbs": round(h_in / t_up / 1e9, 1), "d2h_gbs": round(h_out / t_down / 1e9, 1),
                    "both_gbs": round((h_in + h_out) / t_both / 1e9, 1), "floor_ms_per_step":
                    round(t_both * 1e3, 3)}

        link = link_rates()
        e2e_run(2)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.e2e_steps, args.steps))
        barrier(dist, dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(n_e2e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        et = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, dev)
        code, detail = second["batch"].status(stream)
        if code != 0:
            raise SystemExit(f"bench.py: status {code} detail {detail} in the end-to-end steps")
        e2e = {"value": round(world * sb * n_e2e / et / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h_in), "d2h_bytes_per_step": int(h_out),
               "steps": n_e2e, "ms_per_step": round(et / n_e2e * 1e3, 3),
               "link": dict(link, frac_of_floor=round(link["floor_ms_per_step"] /
                                                      (et / n_e2e * 1e3), 4)),
               "path": "per step: pinned host -> device copies of the full block, miss KV "
                       "and block tables, the step through the C ABI, objects -> pinned host; "
                       "two buffer sets, so one step's copies overlap its neighbours' kernels"}
        del h_hit, h_miss, h_tab, h_obj, sets, second

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(spec, hit=bufs["hit"].cpu().numpy(), miss=bufs["miss"].cpu().numpy())
        cpu = cpu_baseline(spec, args.cpu_seconds, sample)

    if rank == 0:
        cfg = describe(spec)
        cfg.update(layers_per_launch=K,
                   objects="one layer (layer stride 0)" if one_layer else "all layers",
                   hit_layer_buffers=ring,
                   us_per_layer=round(elapsed / args.steps / spec.L * 1e6, 2),
                   layers_per_s=round(world * spec.L * args.steps / elapsed, 1),
                   launch="CUDA graph of one step, replayed per step" if graph is not None
                   else "eager C-ABI calls from Python",
                   kernel_timing="CUDA events around each op's phase of launches (launch "
                   f"duration = phase time / launches), median of {KERNEL_REPS} graph replays "
                   "after the timed region" if graph is not None
                   else "CUDA events around each op's phase of launches, median over the "
                   "timed steps",
                   launch_overlap="none: every launch waits for the one before it"
                   if args.serial_launches else
                   "as below, except gather and scatter-back (shared object layer), "
                   "which run one launch at a time: KVL_LAUNCH_OVERLAP_PREVIOUS on a "
                   "phase's launches after its first, KVL_LAUNCH_SHARE_SMS on the first"
                   if one_layer else
                   "KVL_LAUNCH_OVERLAP_PREVIOUS on a phase's launches after its first "
                   "(each may start beside its predecessor, on half of an SM's shared "
                   "memory), KVL_LAUNCH_SHARE_SMS on the first",
                   step_bytes=sb, kernels=kernels, launches_per_step=launches_per_step,
                   parallelism=f"{world} independent replica(s)", gpu=torch.cuda.get_device_name(dev))
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(elapsed / args.steps * 1e3, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8",
                "data": "synthetic (seeded bf16 KV payload; byte copies)", "config": cfg,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps * world,
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_overlap(args):
    """Layer-wise pipeline under an SM budget: layer l's merge-scatter (at most k CTAs,
    i.e. k SMs) on a transfer stream, and a synthetic compute kernel for layer l (a
    bf16 GEMM standing in for the layer's attention) on a compute stream that waits for
    layer l's transfer.  Transfers run ahead, so layer l+1's copy overlaps layer l's
    compute.  For each budget: the transfer alone, the compute alone, the pipeline, and
    the pipeline's time beyond the compute alone (bubbles plus the slowdown of sharing
    the GPU), next to Tutti's zero-bubble condition T_transfer <= T_compute
    (Tutti 阅读笔记, eq. (17))."""
    import torch
    import layer_wise_paged_gb300 as kvl
    from layer_wise_paged_gb300.batch import Batch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvl.build()
    kvl.lib()
    spec = bench_spec(args)
    bufs = workloads.allocate(spec, dev)
    lay = bufs["layout"]
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    b = Batch(g, lay.requests, bufs["hit"], bufs["miss"], bufs["objects"], bufs["tables"],
              bufs["src_tables"])
    pool = bufs["pool"]
    main = torch.cuda.current_stream(dev)
    b.plan(stream=main)
    n = args.gemm
    A = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    Bm = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    C = torch.empty(n, n, device=dev, dtype=torch.bfloat16)
    xfer, comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    budgets = [k for k in (4, 8, 16, 32, 64, sms) if k <= sms]
    L = spec.L
    per_layer = op_bytes(spec)["merge_scatter"]

    def timed(fn, reps=3):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            fn()
            e1.record(main)
            torch.cuda.synchronize(dev)
            t = e0.elapsed_time(e1) / 1e3
            best = t if best is None else min(best, t)
        return best

    def transfers(k, s):
        for l in range(L):
            b.merge_scatter(l, pool, None, s, max_ctas=k)

    def computes(s):
        for _ in range(L):
            with torch.cuda.stream(s):
                torch.matmul(A, Bm, out=C)

    t_c = timed(lambda: computes(main)) / L
    rows = []
    for k in budgets:
        t_r = timed(lambda: transfers(k, main)) / L

        def pipeline():
            xfer.wait_stream(main)
            comp.wait_stream(main)
            evs = [torch.cuda.Event() for _ in range(L)]
            for l in range(L):
                b.merge_scatter(l, pool, None, xfer, max_ctas=k)
                evs[l].record(xfer)
            for l in range(L):
                comp.wait_event(evs[l])
                with torch.cuda.stream(comp):
                    torch.matmul(A, Bm, out=C)
            main.wait_stream(xfer)
            main.wait_stream(comp)
        t_p = timed(pipeline) / L
        rows.append({"sm_budget": k, "transfer_us_alone": round(t_r * 1e6, 1),
                     "transfer_gbs_alone": round(per_layer / t_r / 1e9, 1),
                     "compute_us_alone": round(t_c * 1e6, 1),
                     "pipeline_us_per_layer": round(t_p * 1e6, 1),
                     "over_compute_frac": round(max(0.0, (t_p - t_c) / t_p), 4),
                     "zero_bubble_alone": bool(t_r <= t_c)})
    code, detail = b.status(main)
    if code != 0:
        raise SystemExit(f"bench.py: status {code} detail {detail}")
    print(json.dumps({"metric": "layer-wise overlap of merge-scatter with compute under an SM budget",
                      "workload": spec.name, "L": L, "gemm": f"bf16 {n}x{n}x{n} per layer",
                      "transfer": "kvl_merge_scatter_paged per layer, at most sm_budget CTAs",
                      "rows": rows}), flush=True)
    return 0


def run_host_leg(args):
    """DualPath's host-buffer legs on one GB300: the full prompt KV held in pinned Grace
    memory, moved over NVLink-C2C.  Fused: merge-scatter of every layer read straight
    from the host full block into the HBM pool (the final H2D and the paging in one
    pass), and gather of every layer's objects straight into host memory.  Against:
    copy-engine copies of the same bytes followed (or preceded) by the device-only op.
    Reported as GB/s across the link and as a fraction of the copy engines' rate."""
    import torch
    import layer_wise_paged_gb300 as kvl
    from layer_wise_paged_gb300.batch import Batch, MappedHost

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvl.build()
    kvl.lib()
    spec = bench_spec(args)
    bufs = workloads.allocate(spec, dev)
    lay = bufs["layout"]
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    main = torch.cuda.current_stream(dev)
    hit_h, miss_h = MappedHost(bufs["hit"].numel()), MappedHost(bufs["miss"].numel())
    obj_h = MappedHost(bufs["objects"].numel())
    hit_h.np[:] = bufs["hit"].cpu().numpy()
    miss_h.np[:] = bufs["miss"].cpu().numpy()
    b_host = Batch(g, lay.requests, hit_h, miss_h, obj_h, bufs["tables"], bufs["src_tables"])
    b_dev = Batch(g, lay.requests, bufs["hit"], bufs["miss"], bufs["objects"], bufs["tables"],
                  bufs["src_tables"])
    b_host.plan(stream=main)
    b_dev.plan(stream=main)
    pool = bufs["pool"]
    L = spec.L
    in_bytes = (sum(spec.t_hit) + sum(spec.t_miss)) * L * spec.R
    obj_bytes = bufs["objects"].numel()
    tin_h = torch.from_numpy(hit_h.np)  # host views for the copy-engine legs
    tmiss_h = torch.from_numpy(miss_h.np)
    tobj_h = torch.from_numpy(obj_h.np)

    def timed(fn, reps=4):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            fn()
            e1.record(main)
            torch.cuda.synchronize(dev)
            t = e0.elapsed_time(e1) / 1e3
            best = t if best is None else min(best, t)
        return best

    H = kvl.KVL_LAUNCH_HOST_SRC
    D = kvl.KVL_LAUNCH_HOST_DST
    t_fused_in = timed(lambda: b_host.merge_scatter(0, pool, None, main, layer_count=L, flags=H))
    t_ce_in = timed(lambda: (bufs["hit"].copy_(tin_h, non_blocking=True),
                             bufs["miss"].copy_(tmiss_h, non_blocking=True)))
    t_dev_merge = timed(lambda: b_dev.merge_scatter(0, pool, None, main, layer_count=L))
    t_fused_out = timed(lambda: b_host.gather(0, pool, main, layer_count=L, flags=D))
    t_dev_gather = timed(lambda: b_dev.gather(0, pool, main, layer_count=L))
    t_ce_out = timed(lambda: tobj_h.copy_(bufs["objects"], non_blocking=True))
    for bt in (b_host, b_dev):
        code, detail = bt.status(main)
        if code != 0:
            raise SystemExit(f"bench.py: status {code} detail {detail}")
    ce_in_gbs, ce_out_gbs = in_bytes / t_ce_in / 1e9, obj_bytes / t_ce_out / 1e9
    print(json.dumps({
        "metric": "host-buffer legs over NVLink-C2C (GB/s across the link)",
        "workload": spec.name, "L": L, "link_bytes_in": in_bytes, "link_bytes_out": obj_bytes,
        "h2d": {"fused_merge_scatter_from_host_gbs": round(in_bytes / t_fused_in / 1e9, 1),
                "copy_engine_gbs": round(ce_in_gbs, 1),
                "copy_engine_then_device_merge_scatter_gbs":
                    round(in_bytes / (t_ce_in + t_dev_merge) / 1e9, 1),
                "fused_frac_of_copy_engine": round(ce_in_gbs and (in_bytes / t_fused_in / 1e9) / ce_in_gbs, 3)},
        "d2h": {"fused_gather_to_host_gbs": round(obj_bytes / t_fused_out / 1e9, 1),
                "copy_engine_gbs": round(ce_out_gbs, 1),
                "device_gather_then_copy_engine_gbs":
                    round(obj_bytes / (t_dev_gather + t_ce_out) / 1e9, 1),
                "fused_frac_of_copy_engine": round((obj_bytes / t_fused_out / 1e9) / ce_out_gbs, 3)},
        "launches": "one launch of all layers per fused leg"}), flush=True)
    return 0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="kvl", choices=["kvl", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.NAMES)
    p.add_argument("--layers", type=int, default=0,
                   help="use only the first N layers of the workload (small profiling case)")
    p.add_argument("--layers-per-launch", type=int, default=1,
                   help="layers each copy launch covers (1 = the layer-wise pipeline)")
    p.add_argument("--objects", default="layer", choices=["layer", "block"],
                   help="object layout: layer-major, or one file per block (2L objects each)")
    p.add_argument("--overlap", action="store_true",
                   help="measure the layer-wise pipeline with compute under SM budgets")
    p.add_argument("--gemm", type=int, default=4096, help="GEMM size of the --overlap compute")
    p.add_argument("--host-leg", action="store_true",
                   help="measure the host-buffer legs over NVLink-C2C")
    p.add_argument("--clocks-csv", default="",
                   help="also write the nvidia-smi clock samples of the timed region here")
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--eager", action="store_true",
                   help="launch every call from Python instead of replaying a CUDA graph")
    p.add_argument("--serial-launches", action="store_true",
                   help="no launch starts before the one before it has finished (no "
                        "KVL_LAUNCH_OVERLAP_PREVIOUS)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be at least 3")
    return a


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.overlap:
        return run_overlap(args)
    if args.host_leg:
        return run_host_leg(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
