"""Benchmark of the layer-wise paged KV block reshuffle on one GB300 (or one batch split
over N GPUs).

One step = the whole hot path over one batch: the batch plan, then for every layer
slice (hit_layer[l]), merge-scatter (hit + miss into the paged pool), gather (pool ->
per-layer K/V objects) and scatter-back (objects -> pool).  The ops run phase by
phase (all layers of one op, then the next op), so no kernel finds its inputs in L2:
every phase streams at least 8 GB through a 129 MB L2.

Prints one JSON line for the headline workload (default: the 256-request batch, the
largest workload that fits one GPU).  `value` is algorithmic bytes moved (read +
write, every op) per second of the timed region, in GB/s; `roofline` is the dominant
kernel's achieved bandwidth against the measured HBM copy peak; `e2e` repeats the
step through the C ABI with the inputs copied from pinned host memory and the objects
read back inside the timed region (and a variant whose slice and merge-scatter read
the pinned host inputs in place); `cpu_baseline` is the CPU oracle on a bounded sample
of the same workload; `serial` is the step with every launch waiting for the one
before it.  `config.per_workload` gives the same step figures for the other full-size
workloads, measured in the same process after the headline, and `host_leg` and
`overlap` the host-buffer legs and the layer-wise pipeline beside compute under an SM
budget, on the Llama-3-8B-shaped turn.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference   # the CPU oracle on the host cores

With N > 1 (one process per GPU under torchrun) the batch is split: each rank takes a
contiguous run of requests (or of layers, for fewer requests than ranks), with its
own pool, plan and objects, and no data-path exchange; `value` is the bytes all ranks
moved over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import contextlib
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
DEFAULT_WORKLOAD = "many_small"
SIDE_WORKLOADS = ("llama3_8b_agentic", "qwen3_32b_long", "latent_batch")
PIPELINE_WORKLOAD = "llama3_8b_agentic"  # host legs and the overlap with compute
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, about 8 TB/s (context for "% of peak")
HIT_RING = 8
E2E_PARTS = 8  # parts of the batch in the staged end-to-end step (one input set)
KERNEL_REPS = 11  # replays whose per-phase events give the per-kernel median
OPS = ("slice", "merge_scatter", "gather", "scatter_back")
KERNEL_NAMES = {"slice": "kvl_slice_kernel", "merge_scatter": "kvl_merge_scatter_kernel",
                "gather": "kvl_gather_kernel", "scatter_back": "kvl_scatter_back_kernel"}
_T0 = time.perf_counter()


def host_available() -> int:
    """Bytes of host memory the kernel reports available (MemAvailable), or 0."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def log(msg: str) -> None:
    """A progress line on stderr (stdout carries only the JSON line)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg} (host memory available "
          f"{host_available() / 1e9:.0f} GB)", file=sys.stderr, flush=True)


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
    if spec.P == 2 and spec.Rp == 2048:
        d.update(H_kv=8, d=128)
    if spec.part:
        d.update(part=spec.part)
    return d


# ---------------------------------------------------------------------------
# Multi-rank plumbing (one process per GPU; the batch split, no data-path collective)
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


def sum_over_ranks(value: float, dist, device=None) -> float:
    """Sum of a value over all ranks (the bytes every rank moved)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_part(spec, world, rank):
    """(Part, its spec) of `rank` when `spec`'s batch is split over `world` GPUs
    (layer_wise_paged_gb300.shard); the spec is None for a rank left idle."""
    from layer_wise_paged_gb300.shard import split_batch
    part = split_batch(spec.t_hit, spec.t_miss, spec.B, spec.L, workloads.block_tables(spec),
                       workloads.source_tables(spec), world, rank)
    return part, workloads.part_spec(spec, part)


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

def phase_launch_flags(op, i, l0, *, ring, n_launches, shared_objects, serial, plan_ready=True):
    """Flags of launch i (first layer l0) of an op's phase of n_launches launches.

    A launch may overlap the one before it only when the two touch disjoint bytes:
    never the first launch of a phase (it reads the previous phase's output), never a
    slice launch that reuses a buffer of the hit_layer ring (l0 a multiple of `ring`),
    and no gather or scatter-back launch when all layers share one layer of objects.
    The launch before a run of overlapping ones leaves them half of each SM.  A launch
    that waits for its predecessor carries KVL_LAUNCH_PLAN_READY (it prefetches while
    that one drains), except the step's first launch, which follows the plan's own
    kernels."""
    from layer_wise_paged_gb300 import (KVL_LAUNCH_OVERLAP_PREVIOUS, KVL_LAUNCH_PLAN_READY,
                                        KVL_LAUNCH_SHARE_SMS)
    ready = KVL_LAUNCH_PLAN_READY if plan_ready and not (op == OPS[0] and i == 0) else 0
    if serial or (shared_objects and op in ("gather", "scatter_back")):
        return ready
    if i == 0 or (op == "slice" and l0 % ring == 0):
        return (KVL_LAUNCH_SHARE_SMS if n_launches > 1 else 0) | ready
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
        """Host bytes one more worker holds while it runs a layer: its own pool and
        objects, plus what one layer's calls allocate while they run (the slice's
        output, and the hit_layer and complete_layer buffers the oracle's merge-scatter
        builds before it scatters)."""
        spec = self.spec
        n_hit, n_all = int(sum(spec.t_hit)), int(spec.t_all().sum())
        return self.pool.nbytes + self.objects.nbytes + (2 * n_hit + n_all) * spec.R

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
    (at most 60 % of the memory available now goes to the workers, each counted with
    everything it holds while it runs a layer)."""
    cores = os.cpu_count() or 1
    want = cores if want is None else max(1, min(int(want), cores))
    avail = host_available()
    if avail <= 0:
        return 1
    return max(1, min(want, int(avail * 0.6 // max(1, sample.worker_bytes()))))


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
    log(f"cpu baseline: {n} oracle threads, {sample.worker_bytes() / 1e9:.1f} GB each")
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
    """The named workload, or its first --layers layers and first --requests requests
    (a smaller case of the same kernels, for profiling captures that must fit in a few
    GB; a batch cut to fewer requests gets a pool of 1.25 times the blocks they use)."""
    spec = workloads.get_spec(args.workload)
    if args.layers:
        spec = dataclasses.replace(spec, L=min(spec.L, args.layers))
    if args.requests and args.requests < spec.n_req:
        n = args.requests
        spec = dataclasses.replace(spec, t_hit=spec.t_hit[:n], t_miss=spec.t_miss[:n])
        spec = dataclasses.replace(spec, n_pool=int(-(-5 * int(spec.nblk().sum()) // 4)))
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
            "scaling": "strong", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
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

    def __init__(self, spec, dev, layers_per_launch=1, serial=False, plan_ready=True):
        import torch
        from layer_wise_paged_gb300.batch import Batch
        self.spec, self.serial, self.plan_ready = spec, serial, plan_ready
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
                                  shared_objects=self.one_layer, serial=self.serial,
                                  plan_ready=self.plan_ready)

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


# ---------------------------------------------------------------------------
# Measurements on one GPU
# ---------------------------------------------------------------------------

def make_event():
    """A timing event that becomes a record node when captured in a CUDA graph (None if
    this torch has no external events)."""
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def check_status(batch, stream, when):
    code, detail = batch.status(stream)
    if code != 0:
        raise SystemExit(f"bench.py: plan status {code} detail {detail} {when}")


def steps_for(spec, seconds, lo=10, hi=200):
    """Steps of `spec` that take about `seconds` at 6.5 TB/s (at least lo, at most hi)."""
    return int(min(hi, max(lo, seconds * 6.5e12 / max(1, step_bytes(spec)))))


def per_op_figures(spec, groups, phase_s):
    """Per-op launch duration (median over samples of phase time / launches), GB/s and
    layers/s, and the dominant op (largest phase time)."""
    per_op = {}
    for op in OPS:
        avg = statistics.median(t / len(groups) for t in phase_s[op])
        per_op[op] = {"us_per_launch": round(avg * 1e6, 2),
                      "gbs": round(op_bytes(spec)[op] * spec.L / len(groups) / avg / 1e9, 1),
                      "layers_per_s": round(spec.L / len(groups) / avg, 1),
                      "total_s": avg * len(groups)}
    dom = max(OPS, key=lambda o: per_op[o]["total_s"])
    return per_op, dom


def measure_step(spec, dev, *, steps, warmup, serial=False, layers_per_launch=1, eager=False,
                 clocks=None, dist=None, kernel_reps=KERNEL_REPS, bs=None, plan_ready=True):
    """`warmup` untimed bench steps of `spec`, then `steps` timed ones (CUDA events on
    the launch stream, max over ranks), each a replay of a CUDA graph of one step (or,
    with `eager`, C-ABI calls from Python).  Per-op launch durations come from events
    around each op's phase of launches: the median of `kernel_reps` replays after the
    timed region (a graph's events hold its last replay), or of the timed steps.
    `bs`: the BenchStep of an earlier measurement of the same workload to reuse (its
    buffers; `serial` and `plan_ready` replace its launch rule), else a new one is
    allocated.
    Returns a dict with the BenchStep (`bs`), `elapsed` (s), `per_op`, `dom` and how
    the step was launched."""
    import torch
    if bs is None:
        bs = BenchStep(spec, dev, layers_per_launch=layers_per_launch, serial=serial)
    bs.serial, bs.plan_ready = serial, plan_ready
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        bs.enqueue(bs.batch, stream)
    torch.cuda.synchronize(dev)
    check_status(bs.batch, stream, "after the warm-up steps")
    graph, ev = None, None
    if not eager and make_event() is not None:
        ev = {op: (make_event(), make_event()) for op in OPS}
        graph = capture_step_graph(dev, stream, lambda s_: bs.enqueue(bs.batch, s_, ev))
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
            bs.enqueue(bs.batch, stream, evs)
            for op in OPS:
                eager_ev[op].append(evs[op])

    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with (clocks if clocks is not None else contextlib.nullcontext()):
        if clocks is not None:
            time.sleep(0.3)
        t0.record(stream)
        for _ in range(steps):
            timed_step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, dist, dev)
    check_status(bs.batch, stream, "after the timed steps")
    if graph is not None:
        phase_s = {op: [] for op in OPS}
        for _ in range(kernel_reps):
            graph.replay()
            torch.cuda.synchronize(dev)
            for op in OPS:
                phase_s[op].append(ev[op][0].elapsed_time(ev[op][1]) / 1e3)
        check_status(bs.batch, stream, "after the timing replays")
    else:
        phase_s = {op: [a.elapsed_time(b) / 1e3 for a, b in eager_ev[op]] for op in OPS}
    per_op, dom = per_op_figures(spec, bs.groups, phase_s)
    del graph
    return dict(bs=bs, elapsed=elapsed, steps=steps, per_op=per_op, dom=dom,
                launch="CUDA graph of one step, replayed per step" if ev is not None
                else "eager C-ABI calls from Python",
                kernel_timing="CUDA events around each op's phase of launches (launch duration "
                f"= phase time / launches), median of {kernel_reps} graph replays after the "
                "timed region" if ev is not None else
                "CUDA events around each op's phase of launches, median over the timed steps")


def dominant_kernel(m):
    """The dominant op's kernel name, with the pipeline depth most of its launches ran
    with (3 stages when sharing SMs with a neighbour launch, else 6)."""
    import layer_wise_paged_gb300 as kvl
    bs, dom = m["bs"], m["dom"]
    shares = bs.flags(dom, 1, bs.groups[1][0]) if len(bs.groups) > 1 else 0
    shares &= kvl.KVL_LAUNCH_OVERLAP_PREVIOUS | kvl.KVL_LAUNCH_SHARE_SMS
    return f"{KERNEL_NAMES[dom]}<{3 if shares else 6}>"


def roofline_of(spec, m, peak, peak_kind):
    """The dominant kernel against the measured copy peak (and the nominal HBM figure);
    traffic from the committed ncu record when it was taken on this kernel source."""
    bs, dom = m["bs"], m["dom"]
    kname = dominant_kernel(m)
    achieved = m["per_op"][dom]["gbs"]
    traffic = recorded_traffic(kname, spec.name) if bs.K == 1 and not spec.part else None
    return {"bound": "hbm", "kernel": kname + f" ({dom})", "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_kind,
            "nominal_peak": NOMINAL_HBM_GBS,
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "algorithmic_bytes_per_launch": op_bytes(spec)[dom] * spec.L // len(bs.groups),
            "traffic": traffic,
            "traffic_source": "profiles/dram_traffic.txt (ncu dram__bytes_read.sum + "
                              "dram__bytes_write.sum per launch, this kernel source)"
            if traffic is not None else None}


def step_summary(spec, m, peak):
    """The figures of one measured step: GB/s, µs per layer, per-op kernels, the
    dominant kernel's fraction of the measured and nominal peaks."""
    sb = step_bytes(spec)
    gbs = sb * m["steps"] / m["elapsed"] / 1e9
    dom = m["dom"]
    return {"step_gbs": round(gbs, 1), "ms_per_step": round(m["elapsed"] / m["steps"] * 1e3, 4),
            "us_per_layer": round(m["elapsed"] / m["steps"] / spec.L * 1e6, 2),
            "layers_per_s": round(spec.L * m["steps"] / m["elapsed"], 1), "steps": m["steps"],
            "step_frac": round(gbs / peak, 4),
            "kernels": {op: {k: v for k, v in m["per_op"][op].items() if k != "total_s"}
                        for op in OPS},
            "dominant": dominant_kernel(m) + f" ({dom})",
            "frac": round(m["per_op"][dom]["gbs"] / peak, 4),
            "frac_of_nominal": round(m["per_op"][dom]["gbs"] / NOMINAL_HBM_GBS, 4)}


def request_parts(spec, k):
    """The batch as at most k contiguous request ranges [a, z), none empty, balanced by
    each request's step bytes with the batch split's midpoint rule."""
    from layer_wise_paged_gb300.shard import request_weights, split_requests
    n = spec.n_req
    k = max(1, min(int(k), n))
    if k == 1:
        return [(0, n)]
    ranks = split_requests(request_weights(spec.t_hit, spec.t_miss, spec.B), k)
    cuts = [0] + [int(np.searchsorted(ranks, r)) for r in range(1, k)] + [n]
    return [(a, z) for a, z in zip(cuts[:-1], cuts[1:]) if z > a]


class EndToEnd:
    """The bench step through the C ABI with its inputs in pinned host memory (Grace
    memory, over NVLink-C2C) and its objects read back to pinned host memory, every
    step, inside the timed region.  Two variants:

    * staged: per step, copy-engine copies of the block tables, the full block and
      the miss KV into HBM, then the step, with each gathered layer of objects copied
      back to the host as soon as it exists;
    * in place: the same, except that the slice and merge-scatter read the full block
      and the miss KV straight from pinned host memory (KVL_LAUNCH_HOST_SRC: SM loads
      over the link), so nothing is staged in HBM first.

    Launches are eager C-ABI calls from Python; copies run on their own streams.
    Uploads overlap kernels in one of two ways:

    * two device input sets, where device memory allows: a step's uploads go to the set
      the step before last used, once that step's merge-scatter is done with it;
    * otherwise the batch runs as `parts` parts of its requests (contiguous runs split
      by bytes, over the same buffers), one after the other, each part with its own
      launches: a part's uploads wait only for that part's merge-scatter of the step
      before, so they run while the other parts' kernels run.

    Object buffers are slots that a gather waits on only until its last read-back of
    that slot is done.  With all layers in one object buffer each input set has its
    own; when all layers share one object layer (the largest workloads), the gathers
    rotate over a ring of `ring` such layers, so read-backs trail the gathers, and
    scatter-back of layer l reads slot l mod ring.  Each part reads back only its own
    requests' bytes of a slot.  Each (set, part, slot) has its own batch and plan; a
    step builds all of its plans before its first copy launch."""

    def __init__(self, bs, dev, ring=4, two_sets=True, parts=None):
        import torch
        from layer_wise_paged_gb300.batch import Batch, MappedHost
        self.bs, self.dev = bs, dev
        b = bs.bufs
        n_obj = b["objects"].numel()
        host_slots = 2 if bs.one_layer else 1
        need = b["hit"].numel() + b["miss"].numel() + host_slots * n_obj
        avail = host_available()
        if need > 0.6 * avail:
            raise MemoryError(f"pinned host buffers of {need / 1e9:.0f} GB, host memory "
                              f"available {avail / 1e9:.0f} GB")
        log(f"end to end: pinning {need / 1e9:.1f} GB of host memory")
        self.h_hit = MappedHost(b["hit"].numel())
        self.h_miss = MappedHost(b["miss"].numel())
        self.h_obj = [MappedHost(n_obj) for _ in range(host_slots)]
        log("end to end: host buffers pinned")
        self.t_hit = torch.from_numpy(self.h_hit.np)[:b["hit"].numel()]
        self.t_miss = torch.from_numpy(self.h_miss.np)[:b["miss"].numel()]
        self.t_hit.copy_(b["hit"])
        self.t_miss.copy_(b["miss"])
        self.h_tab = torch.empty(b["tables"].numel(), dtype=torch.int32, pin_memory=True)
        self.h_tab.copy_(b["tables"])
        log("end to end: host inputs written")
        self.t_obj = [torch.from_numpy(h.np)[:n_obj] for h in self.h_obj]
        spec, lay = bs.spec, b["layout"]
        g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
        # device input sets: the bench's own, and a second one where memory allows
        second = b["hit"].numel() + b["miss"].numel() + (0 if bs.one_layer else n_obj)
        self.n_sets = 2 if two_sets and second + 16e9 < torch.cuda.mem_get_info(dev)[0] else 1
        self.sets = [dict(hit=b["hit"], miss=b["miss"], tables=b["tables"])]
        if self.n_sets == 2:
            self.sets.append(dict(hit=torch.empty_like(b["hit"]), miss=torch.empty_like(b["miss"]),
                                  tables=torch.empty_like(b["tables"])))
        # object slots: a ring of shared object layers, or one buffer per input set
        self.ring = max(1, min(int(ring), spec.L)) if bs.one_layer else self.n_sets
        self.d_obj = [b["objects"]] + [torch.full_like(b["objects"], workloads.SENTINEL)
                                       for _ in range(self.ring - 1)]
        # parts of the batch (one input set only): request ranges split by bytes
        n = spec.n_req
        bounds = request_parts(spec, E2E_PARTS if parts is None else parts) \
            if self.n_sets == 1 else [(0, n)]
        blk_off = np.concatenate([[0], np.cumsum(spec.nblk())]).astype(np.int64)
        hit_rows = np.concatenate([[0], np.cumsum(np.asarray(spec.t_hit, np.int64))])
        reqs = lay.requests

        def edge(i, field, total):
            return getattr(reqs[i], field) if i < n else total

        self.parts = []
        for i0, i1 in bounds:
            part = dict(reqs=reqs[i0:i1], hit=(edge(i0, "hit_off", lay.hit_bytes),
                                               edge(i1, "hit_off", lay.hit_bytes)),
                        miss=(edge(i0, "miss_off", lay.miss_bytes), edge(i1, "miss_off", lay.miss_bytes)),
                        obj=(edge(i0, "obj_off", lay.obj_bytes), edge(i1, "obj_off", lay.obj_bytes)),
                        tab=(int(blk_off[i0]), int(blk_off[i1])), hit_row0=int(hit_rows[i0]))
            t0, t1 = part["tab"]
            part["dev"] = [[Batch(g, part["reqs"], st["hit"], st["miss"], o, st["tables"][t0:t1],
                                  b["src_tables"]) for o in self.d_obj] for st in self.sets]
            part["host"] = [Batch(g, part["reqs"], self.h_hit, self.h_miss, o, b["tables"][t0:t1],
                                  b["src_tables"]) for o in self.d_obj]
            self.parts.append(part)
        # the whole batch over the host inputs (the host legs use it)
        self.b_host = Batch(g, reqs, self.h_hit, self.h_miss, self.d_obj[0], b["tables"],
                            b["src_tables"])
        self.main = torch.cuda.current_stream(dev)
        self.h2d, self.d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        self.ev_g = torch.cuda.Event()
        keys = [(si, pi) for si in range(self.n_sets) for pi in range(len(self.parts))]
        self.ev_tab = [torch.cuda.Event() for _ in range(self.n_sets)]  # a set's tables in place
        self.ev_in = {k: torch.cuda.Event() for k in keys}              # a region's inputs in place
        self.ev_free = {k: torch.cuda.Event() for k in keys}            # a region's inputs done with
        self.ev_slot = {(pi, k): torch.cuda.Event() for pi in range(len(self.parts))
                        for k in range(self.ring)}                      # a part's slot read back
        self.n_step = 0
        self.used = set()  # the batches steps have planned and used (their status is read)
        self.h2d_bytes = b["hit"].numel() + b["miss"].numel() + 4 * b["tables"].numel()
        self.reads_back = spec.L if bs.one_layer else 1
        self.d2h_bytes = n_obj * self.reads_back
        # bytes the in-place slice and merge-scatter read across the link per step
        self.in_place_bytes = (op_bytes(spec)["slice"] + op_bytes(spec)["merge_scatter"]) // 2 * spec.L

    def _read_back(self, pi, slot, host_slot):
        import torch
        o0, o1 = self.parts[pi]["obj"]
        self.ev_g.record(self.main)
        self.d2h.wait_event(self.ev_g)
        with torch.cuda.stream(self.d2h):
            self.t_obj[host_slot][o0:o1].copy_(self.d_obj[slot][o0:o1], non_blocking=True)
        self.ev_slot[(pi, slot)].record(self.d2h)

    def _step(self, in_place):
        import torch
        import layer_wise_paged_gb300 as kvl
        bs, s = self.bs, self.main
        si = 0 if in_place else self.n_step % self.n_sets
        own = self.n_step % self.ring
        self.n_step += 1
        st = self.sets[si]
        # the slot of each layer's gather: a ring position, or the step's own buffer
        slot_of = (lambda i: i % self.ring) if bs.one_layer else (lambda i: own)
        # uploads: the tables once the step that last used this set has planned (its
        # first part's merge-scatter is later still), then each part's inputs once that
        # part's merge-scatter of the step before is done with them
        self.h2d.wait_event(self.ev_free[(si, 0)])
        with torch.cuda.stream(self.h2d):
            st["tables"].copy_(self.h_tab, non_blocking=True)
        self.ev_tab[si].record(self.h2d)
        for pi, part in enumerate(self.parts):
            if in_place:
                break
            self.h2d.wait_event(self.ev_free[(si, pi)])
            (h0, h1), (m0, m1) = part["hit"], part["miss"]
            with torch.cuda.stream(self.h2d):
                st["hit"][h0:h1].copy_(self.t_hit[h0:h1], non_blocking=True)
                st["miss"][m0:m1].copy_(self.t_miss[m0:m1], non_blocking=True)
            self.ev_in[(si, pi)].record(self.h2d)
        # every plan of the step first, so that each copy launch after them follows a
        # complete plan
        s.wait_event(self.ev_tab[si])
        slots = sorted({slot_of(i) for i in range(len(bs.groups))})
        for part in self.parts:
            rows = part["host"] if in_place else part["dev"][si]
            for k in slots:
                rows[k].plan(stream=s)
                self.used.add(rows[k])
        host = kvl.KVL_LAUNCH_HOST_SRC
        layer_hit = bs.layer_hit
        for pi, part in enumerate(self.parts):
            rows = part["host"] if in_place else part["dev"][si]
            if not in_place:
                s.wait_event(self.ev_in[(si, pi)])
            batch = rows[slot_of(0)]
            off = part["hit_row0"] * bs.spec.R
            for i, (l0, n) in enumerate(bs.groups):
                hv = bs.hit_out[(l0 % bs.ring) * layer_hit + off:]
                batch.slice_layer(l0, hv, s, layer_count=n,
                                  flags=host if in_place else bs.flags("slice", i, l0))
            for i, (l0, n) in enumerate(bs.groups):
                batch.merge_scatter(l0, bs.pool, None, s, layer_count=n,
                                    flags=host if in_place else bs.flags("merge_scatter", i, l0))
            self.ev_free[(si, pi)].record(s)
            for i, (l0, n) in enumerate(bs.groups):
                k = slot_of(i)
                if bs.one_layer or i == 0:
                    s.wait_event(self.ev_slot[(pi, k)])  # this part's last read-back of the slot
                rows[k].gather(l0, bs.pool, s, layer_count=n, flags=bs.flags("gather", i, l0))
                if bs.one_layer:
                    self._read_back(pi, k, i % 2)
            if not bs.one_layer:
                self._read_back(pi, slot_of(0), 0)
            for i, (l0, n) in enumerate(bs.groups):
                rows[slot_of(i)].scatter_back(l0, bs.pool, s, layer_count=n,
                                              flags=bs.flags("scatter_back", i, l0))

    def status_ok(self) -> bool:
        """Every batch the steps used reports no error (reads back, synchronising)."""
        return all(bt.status(self.main) == (0, 0) for bt in self.used)

    def run(self, n, in_place):
        """n steps; returns seconds (CUDA events on the launch stream)."""
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(self.dev)
        e0.record(self.main)
        for ev in list(self.ev_free.values()) + list(self.ev_slot.values()):
            ev.record(self.main)
        for _ in range(n):
            self._step(in_place)
        self.main.wait_stream(self.h2d)
        self.main.wait_stream(self.d2h)
        e1.record(self.main)
        torch.cuda.synchronize(self.dev)
        for bt in self.used:
            check_status(bt, self.main, "in the end-to-end steps")
        return e0.elapsed_time(e1) / 1e3

    def link_rates(self, reps=2):
        """The copy engines' rates on this machine for the step's own transfers: inputs in
        alone, objects out alone (as the step reads them back), and both at once, each
        timed as whole-buffer copies and as the step's per-part copies; the faster of
        the two counts."""
        import torch
        b = self.bs.bufs

        def timed(fn):
            best = None
            for _ in range(reps):
                torch.cuda.synchronize(self.dev)
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(self.main)
                self.h2d.wait_stream(self.main)
                self.d2h.wait_stream(self.main)
                fn()
                self.main.wait_stream(self.h2d)
                self.main.wait_stream(self.d2h)
                z.record(self.main)
                torch.cuda.synchronize(self.dev)
                t = a.elapsed_time(z) / 1e3
                best = t if best is None else min(best, t)
            return best

        whole = [dict(hit=(0, b["hit"].numel()), miss=(0, b["miss"].numel()),
                      obj=(0, self.d_obj[0].numel()))]

        def up(parts):
            with torch.cuda.stream(self.h2d):
                b["tables"].copy_(self.h_tab, non_blocking=True)
                for part in parts:
                    (h0, h1), (m0, m1) = part["hit"], part["miss"]
                    b["hit"][h0:h1].copy_(self.t_hit[h0:h1], non_blocking=True)
                    b["miss"][m0:m1].copy_(self.t_miss[m0:m1], non_blocking=True)

        def down(parts):
            with torch.cuda.stream(self.d2h):
                for k in range(self.reads_back):
                    for part in parts:
                        o0, o1 = part["obj"]
                        self.t_obj[k % len(self.t_obj)][o0:o1].copy_(
                            self.d_obj[k % self.ring][o0:o1], non_blocking=True)

        pats = [whole] + ([self.parts] if len(self.parts) > 1 else [])
        t_up = min(timed(lambda: up(p)) for p in pats)
        t_down = min(timed(lambda: down(p)) for p in pats)
        t_both = min(timed(lambda: (up(p), down(p))) for p in pats)
        return {"h2d_gbs": round(self.h2d_bytes / t_up / 1e9, 1),
                "d2h_gbs": round(self.d2h_bytes / t_down / 1e9, 1),
                "both_gbs": round((self.h2d_bytes + self.d2h_bytes) / t_both / 1e9, 1),
                "floor_ms_per_step": round(t_both * 1e3, 3)}

    @staticmethod
    def floor_s(link, bytes_in, bytes_out):
        """The least time the link allows for these bytes at the copy engines' measured
        rates: each direction alone, and both together."""
        return max(bytes_in / (link["h2d_gbs"] * 1e9), bytes_out / (link["d2h_gbs"] * 1e9),
                   (bytes_in + bytes_out) / (link["both_gbs"] * 1e9))

    def measure(self, steps, dist=None):
        """Both variants: link rates first, a warm-up step each, then `steps` timed
        steps each.  Returns the e2e JSON object (staged as the headline).  With several
        ranks the bytes are every rank's and the time the slowest rank's."""
        spec = self.bs.spec
        ranks = 1 if dist is None else dist.get_world_size()
        sb = sum_over_ranks(float(step_bytes(spec)), dist, self.dev)
        before = self.link_rates()
        runs = {}
        for name, in_place in (("staged", False), ("in_place", True)):
            self.run(1, in_place)
            barrier(dist, self.dev)
            runs[name] = max_over_ranks(self.run(steps, in_place), dist, self.dev)
        after = self.link_rates()
        # the link's rate drifts on some boxes: the floor takes the faster of the two
        # measurements on each side of the timed steps, so a slow spell cannot lower it
        link = {k: max(before[k], after[k]) for k in ("h2d_gbs", "d2h_gbs", "both_gbs")}
        link["floor_ms_per_step"] = min(before["floor_ms_per_step"], after["floor_ms_per_step"])
        link["before"], link["after"] = before, after
        out = {}
        for name, in_place in (("staged", False), ("in_place", True)):
            t = runs[name]
            link_in = (self.in_place_bytes + 4 * self.bs.bufs["tables"].numel()) if in_place \
                else self.h2d_bytes
            floor = link["floor_ms_per_step"] / 1e3 if not in_place else \
                self.floor_s(link, link_in, self.d2h_bytes)
            link_all = sum_over_ranks(float(link_in + self.d2h_bytes), dist, self.dev)
            out[name] = {"value": round(sb * steps / t / 1e9, 2), "unit": UNIT,
                         "link_gbs": round(link_all * steps / t / 1e9, 1),
                         "ms_per_step": round(t / steps * 1e3, 3), "steps": steps,
                         "link_in_bytes_per_step": int(link_in),
                         "link_out_bytes_per_step": int(self.d2h_bytes)}
            if in_place:
                # its inputs cross by SM loads, which can beat the copy engines' rates
                out[name].update(copy_engine_floor_ms_per_step=round(floor * 1e3, 3),
                                 frac_of_copy_engine_floor=round(floor / (t / steps), 4))
            else:
                out[name].update(floor_ms_per_step=round(floor * 1e3, 3),
                                 frac_of_floor=round(floor / (t / steps), 4))
        st = out["staged"]
        h2d = int(sum_over_ranks(float(self.h2d_bytes), dist, self.dev))
        d2h = int(sum_over_ranks(float(self.d2h_bytes), dist, self.dev))
        return {"value": st["value"], "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": steps, "ranks": ranks,
                "ms_per_step": st["ms_per_step"], "link_gbs": st["link_gbs"],
                "value_meaning": "HBM-algorithmic bytes of the step (as `value`) per second "
                                 "of the end-to-end step; link_gbs = bytes across the host "
                                 "link per second",
                "link": dict(link, frac_of_floor=st["frac_of_floor"]),
                "in_place": out["in_place"],
                "path": "per step: pinned host -> device copies of the block tables, full "
                        "block and miss KV, the step through the C ABI (eager calls), each "
                        "gathered layer's objects -> pinned host as soon as it exists"
                        + (f" (a ring of {self.ring} device object layers, one plan each, "
                           "two host slots)" if self.bs.one_layer else " (all layers in one copy)")
                        + (f"; {self.n_sets} device input sets used in turn" if self.n_sets > 1
                           else f"; the batch in {len(self.parts)} parts of its requests, "
                                "each part's uploads overlapping the other parts' kernels"
                           if len(self.parts) > 1 else "")
                        + "; in_place: the slice and merge-scatter read the host full block "
                          "and miss KV in place (KVL_LAUNCH_HOST_SRC), nothing staged"}

    def close(self):
        for h in [self.h_hit, self.h_miss] + self.h_obj:
            h.__del__()
        self.t_hit = self.t_miss = self.t_obj = self.h_obj = None
        self.d_obj = self.parts = self.b_host = self.sets = self.used = None


def measure_host_leg(bs, e2e, dev):
    """DualPath's host-buffer legs on one GB300 (host buffers in Grace memory, over
    NVLink-C2C): the merge-scatter of every layer read straight from the pinned host
    full block into the HBM pool (the final H2D and the paging in one pass), and the
    gather of every layer's objects straight into pinned host memory; each against the
    copy engines moving the same bytes.  GB/s across the link."""
    import torch
    import layer_wise_paged_gb300 as kvl
    from layer_wise_paged_gb300.batch import Batch
    spec, b = bs.spec, bs.bufs
    if bs.one_layer:
        raise ValueError("the host legs need a workload whose objects hold every layer")
    main = torch.cuda.current_stream(dev)
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    b_out = Batch(g, b["layout"].requests, b["hit"], b["miss"], e2e.h_obj[0], b["tables"],
                  b["src_tables"])
    e2e.b_host.plan(stream=main)
    b_out.plan(stream=main)
    bs.batch.plan(stream=main)
    L = spec.L
    in_bytes = (sum(spec.t_hit) + sum(spec.t_miss)) * L * spec.R
    obj_bytes = b["objects"].numel()

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

    H, D = kvl.KVL_LAUNCH_HOST_SRC, kvl.KVL_LAUNCH_HOST_DST
    t_fused_in = timed(lambda: e2e.b_host.merge_scatter(0, bs.pool, None, main, layer_count=L, flags=H))
    t_ce_in = timed(lambda: (b["hit"].copy_(e2e.t_hit, non_blocking=True),
                             b["miss"].copy_(e2e.t_miss, non_blocking=True)))
    t_fused_out = timed(lambda: b_out.gather(0, bs.pool, main, layer_count=L, flags=D))
    t_ce_out = timed(lambda: e2e.t_obj[0].copy_(b["objects"], non_blocking=True))
    for bt in (e2e.b_host, b_out):
        check_status(bt, main, "in the host legs")
    fin, fout = in_bytes / t_fused_in / 1e9, obj_bytes / t_fused_out / 1e9
    cin, cout = in_bytes / t_ce_in / 1e9, obj_bytes / t_ce_out / 1e9
    return {"workload": spec.name, "h2d_gbs": round(fin, 1), "d2h_gbs": round(fout, 1),
            "copy_engine_h2d_gbs": round(cin, 1), "copy_engine_d2h_gbs": round(cout, 1),
            "frac_of_link": {"h2d": round(fin / cin, 3), "d2h": round(fout / cout, 3)},
            "link_bytes": {"h2d": int(in_bytes), "d2h": int(obj_bytes)},
            "legs": "h2d: merge-scatter of all layers in one launch, reading the pinned host "
                    "full block and miss KV (KVL_LAUNCH_HOST_SRC); d2h: gather of all layers "
                    "in one launch into pinned host objects (KVL_LAUNCH_HOST_DST); "
                    "frac_of_link = fused rate / copy-engine rate for the same bytes"}


def measure_overlap(bs, dev, gemm=8192, budgets=(4, 8, 16, 32, 64)):
    """Layer-wise pipeline under an SM budget: layer l's merge-scatter (at most k CTAs,
    so at most k SMs) on a transfer stream, and a synthetic compute kernel for layer l
    (a bf16 GEMM standing in for the layer's attention) on a compute stream that waits
    for layer l's transfer.  Transfers run ahead, so layer l+1's copy overlaps layer
    l's compute.  Per budget: the transfer alone, the compute alone, the pipeline, the
    pipeline's slowdown against the compute alone, and Tutti's zero-bubble condition
    T_transfer <= T_compute (Tutti 阅读笔记, eq. (17))."""
    import torch
    spec, b, pool = bs.spec, bs.batch, bs.pool
    main = torch.cuda.current_stream(dev)
    b.plan(stream=main)
    A = torch.randn(gemm, gemm, device=dev, dtype=torch.bfloat16)
    Bm = torch.randn(gemm, gemm, device=dev, dtype=torch.bfloat16)
    C = torch.empty(gemm, gemm, device=dev, dtype=torch.bfloat16)
    xfer, comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
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

    def computes():
        for _ in range(L):
            torch.matmul(A, Bm, out=C)

    t_c = timed(computes) / L
    rows = []
    for k in [k for k in budgets if k < sms] + [sms]:
        t_r = timed(lambda: [b.merge_scatter(l, pool, None, main, max_ctas=k) for l in range(L)]) / L

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
        rows.append({"sm_budget": k, "t_transfer_us": round(t_r * 1e6, 1),
                     "transfer_gbs": round(per_layer / t_r / 1e9, 1),
                     "t_compute_us": round(t_c * 1e6, 1), "pipeline_us": round(t_p * 1e6, 1),
                     "gemm_slowdown_pct": round(100.0 * (t_p - t_c) / t_c, 2),
                     "zero_bubble": bool(t_r <= t_c)})
    check_status(b, main, "in the overlap measurement")
    ok = [r for r in rows if r["zero_bubble"]]
    best = min(ok, key=lambda r: r["sm_budget"]) if ok else None
    return {"workload": spec.name, "gemm": f"bf16 {gemm}x{gemm}x{gemm} per layer",
            "transfer": "kvl_merge_scatter_paged per layer, at most sm_budget CTAs",
            "sm_budget": best["sm_budget"] if best else None,
            "gemm_slowdown_pct": best["gemm_slowdown_pct"] if best else None,
            "t_transfer_us": best["t_transfer_us"] if best else None,
            "t_compute_us": round(t_c * 1e6, 1),
            "summary": "smallest SM budget whose transfer alone meets the zero-bubble "
                       "condition, with the pipeline's slowdown against the compute alone",
            "rows": rows}


def run_gpu(args):
    import torch
    import layer_wise_paged_gb300 as kvl

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    kvl.build()
    kvl.lib()
    peak, peak_kind = hbm_peak()

    whole = bench_spec(args)
    log(f"workload {whole.name}: {step_bytes(whole) / 1e9:.1f} GB per step")
    part, spec = (None, whole) if world == 1 else rank_part(whole, world, rank)
    if world > 1:
        # every rank works out every rank's part (host arithmetic), so that all of them
        # stop together, before any collective, if one would be left without work
        idle = [r for r in range(world) if rank_part(whole, world, r)[1] is None]
        if idle:
            raise SystemExit(f"bench.py: ranks {idle} of {world} would have no part of "
                             f"{whole.name} (more ranks than requests and layers)")
    clk = ClockSampler(local, Path(args.clocks_csv) if args.clocks_csv else None)
    ready = not args.no_plan_ready
    m = measure_step(spec, dev, steps=args.steps, warmup=args.warmup,
                     serial=args.serial_launches, layers_per_launch=args.layers_per_launch,
                     eager=args.eager, clocks=clk, dist=dist, plan_ready=ready)
    bs = m["bs"]
    log(f"headline step measured: {step_bytes(spec) * args.steps / m['elapsed'] / 1e9:.0f} GB/s")
    one_layer, n_groups = bs.one_layer, len(bs.groups)
    sb = step_bytes(spec)
    total_bytes = sum_over_ranks(float(sb * args.steps), dist, dev)
    value = total_bytes / m["elapsed"] / 1e9
    summ = step_summary(spec, m, peak)
    roofline = roofline_of(spec, m, peak, peak_kind)
    launches_per_step = kvl.kvl_launches_per_call(0) + n_groups * 4

    e2e = None
    cpu = None
    ee = None
    if not args.no_e2e:
        try:
            ee = EndToEnd(bs, dev, two_sets=args.e2e_sets == 2, parts=args.e2e_parts)
        except MemoryError as exc:
            e2e = {"skipped": str(exc)}
            log(f"end to end skipped: {exc}")
    if ee is not None:
        e2e = ee.measure(max(3, min(args.e2e_steps, args.steps)), dist)
        log(f"end to end measured: {e2e['value']} GB/s, in place {e2e['in_place']['value']} GB/s")
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            # the oracle reads the same host inputs the end-to-end step uploads
            sample = OracleSample(spec, hit=ee.h_hit.np, miss=ee.h_miss.np)
            cpu = cpu_baseline(spec, args.cpu_seconds, sample)
            log(f"cpu baseline measured: {cpu['value']} GB/s on {cpu['cores']} threads")
            del sample
        ee.close()
        del ee
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(spec, hit=bs.bufs["hit"].cpu().numpy(),
                              miss=bs.bufs["miss"].cpu().numpy())
        cpu = cpu_baseline(spec, args.cpu_seconds, sample)
        del sample

    extras = world == 1 and not args.no_extras
    serial = None
    if extras and not args.serial_launches:
        ms = measure_step(spec, dev, steps=steps_for(spec, 2.0, lo=5, hi=args.steps), warmup=3,
                          serial=True, layers_per_launch=args.layers_per_launch, bs=bs,
                          plan_ready=ready)
        serial = dict(step_summary(spec, ms, peak),
                      launches="every launch waits for the one before it (no "
                               "KVL_LAUNCH_OVERLAP_PREVIOUS)")
        log(f"serial step measured: {serial['step_gbs']} GB/s")
        del ms
    del bs, m["bs"]
    torch.cuda.empty_cache()

    per_workload, host_leg, overlap = {}, None, None
    if extras:
        for name in [n for n in SIDE_WORKLOADS if n != spec.name]:
            side = workloads.get_spec(name)
            free = torch.cuda.mem_get_info(dev)[0]
            need = workloads.footprint_bytes(side, objects_one_layer=workloads.footprint_bytes(side) > 160e9)
            if need + 24e9 > free:
                per_workload[name] = {"skipped": f"needs {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free"}
                continue
            log(f"{name}: allocating {need / 1e9:.0f} GB")
            ms = measure_step(side, dev, steps=steps_for(side, 1.0), warmup=3, plan_ready=ready)
            entry = step_summary(side, ms, peak)
            log(f"{name}: step {entry['step_gbs']} GB/s")
            bs2 = ms.pop("bs")
            keep = ("step_gbs", "us_per_layer", "step_frac", "frac", "dominant", "kernels")
            mser = measure_step(side, dev, steps=steps_for(side, 1.0), warmup=3, serial=True,
                                bs=bs2, plan_ready=ready)
            entry["serial"] = {k: v for k, v in step_summary(side, mser, peak).items() if k in keep}
            if name == PIPELINE_WORKLOAD and ready:
                # the same lone launches without the prefetch ahead of the wait
                m0 = measure_step(side, dev, steps=steps_for(side, 1.0), warmup=3, serial=True,
                                  bs=bs2, plan_ready=False)
                entry["serial_without_plan_ready"] = {
                    k: v for k, v in step_summary(side, m0, peak).items() if k in keep}
                del m0["bs"]
            del mser["bs"]
            if name == PIPELINE_WORKLOAD and not args.no_e2e:
                bs2.serial = False
                ee = EndToEnd(bs2, dev, two_sets=args.e2e_sets == 2, parts=args.e2e_parts)
                e = ee.measure(steps_for(side, 0.5, lo=5, hi=30))
                entry["e2e"] = {k: e[k] for k in ("value", "link_gbs", "ms_per_step",
                                                  "h2d_bytes_per_step", "d2h_bytes_per_step",
                                                  "link", "in_place")}
                host_leg = measure_host_leg(bs2, ee, dev)
                log(f"{name}: host legs {host_leg['h2d_gbs']} / {host_leg['d2h_gbs']} GB/s")
                overlap = measure_overlap(bs2, dev, gemm=args.gemm)
                log(f"{name}: overlap measured")
                ee.close()
                del ee
            del bs2
            per_workload[name] = entry
            torch.cuda.empty_cache()

    if rank == 0:
        cfg = describe(whole if world > 1 else spec)
        cfg.update(layers_per_launch=args.layers_per_launch,
                   objects="one layer (layer stride 0)" if one_layer else "all layers",
                   hit_layer_buffers=HIT_RING,
                   us_per_layer=round(m["elapsed"] / args.steps / spec.L * 1e6, 2),
                   layers_per_s=round(spec.L * args.steps / m["elapsed"], 1),
                   launch=m["launch"], kernel_timing=m["kernel_timing"],
                   launch_overlap="none: every launch waits for the one before it"
                   if args.serial_launches else
                   "KVL_LAUNCH_OVERLAP_PREVIOUS on a phase's launches after its first (each "
                   "may start beside its predecessor, on half of an SM's shared memory), "
                   "KVL_LAUNCH_SHARE_SMS on the first; gather and scatter-back one launch "
                   "at a time when all layers share one object layer",
                   step_bytes=sb, kernels=summ["kernels"], launches_per_step=launches_per_step,
                   parallelism="1 GPU" if world == 1 else
                   f"{world} ranks, one batch split ({part.kind} per rank), no data-path exchange",
                   gpu=torch.cuda.get_device_name(dev), per_workload=per_workload)
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(m["elapsed"] / args.steps * 1e3, 4), "higher_is_better": True,
                "scaling": "strong", "vs_baseline": None, "dtype": "u8",
                "data": "synthetic (seeded bf16 KV payload; byte copies)", "config": cfg,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "serial": serial,
                "host_leg": host_leg, "overlap": overlap,
                "gpu_launches": launches_per_step * args.steps * world,
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_overlap(args):
    """The overlap measurement alone, on --workload, as its own JSON line."""
    import torch
    import layer_wise_paged_gb300 as kvl
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvl.build()
    kvl.lib()
    bs = BenchStep(bench_spec(args), dev)
    print(json.dumps(dict(measure_overlap(bs, dev, gemm=args.gemm),
                          metric="layer-wise overlap of merge-scatter with compute under an SM "
                                 "budget")), flush=True)
    return 0


def run_host_leg(args):
    """The host-buffer legs alone, on --workload, as their own JSON line."""
    import torch
    import layer_wise_paged_gb300 as kvl
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvl.build()
    kvl.lib()
    bs = BenchStep(bench_spec(args), dev)
    ee = EndToEnd(bs, dev)
    print(json.dumps(dict(measure_host_leg(bs, ee, dev),
                          metric="host-buffer legs over NVLink-C2C (GB/s across the link)")),
          flush=True)
    ee.close()
    return 0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="kvl", choices=["kvl", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=workloads.NAMES)
    p.add_argument("--layers", type=int, default=0,
                   help="use only the first N layers of the workload (small profiling case)")
    p.add_argument("--requests", type=int, default=0,
                   help="use only the first N requests of the workload (small profiling case)")
    p.add_argument("--layers-per-launch", type=int, default=1,
                   help="layers each copy launch covers (1 = the layer-wise pipeline)")
    p.add_argument("--objects", default="layer", choices=["layer", "block"],
                   help="object layout: layer-major, or one file per block (2L objects each)")
    p.add_argument("--overlap", action="store_true",
                   help="only measure the layer-wise pipeline with compute under SM budgets")
    p.add_argument("--gemm", type=int, default=8192, help="GEMM size of the overlap compute")
    p.add_argument("--host-leg", action="store_true",
                   help="only measure the host-buffer legs over NVLink-C2C")
    p.add_argument("--clocks-csv", default="",
                   help="also write the nvidia-smi clock samples of the timed region here")
    p.add_argument("--e2e-steps", type=int, default=4)
    p.add_argument("--e2e-sets", type=int, default=2, choices=[1, 2],
                   help="device input sets the staged end-to-end step alternates (2 where "
                        "memory allows)")
    p.add_argument("--e2e-parts", type=int, default=E2E_PARTS,
                   help="with one device input set, the staged end-to-end step runs the batch "
                        "as this many byte-balanced parts of its requests")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the serial step, the other workloads, the host legs and the "
                        "overlap measurement")
    p.add_argument("--eager", action="store_true",
                   help="launch every call from Python instead of replaying a CUDA graph")
    p.add_argument("--serial-launches", action="store_true",
                   help="no launch starts before the one before it has finished (no "
                        "KVL_LAUNCH_OVERLAP_PREVIOUS)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-plan-ready", action="store_true",
                   help="no KVL_LAUNCH_PLAN_READY: launches that wait prefetch nothing first")
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
