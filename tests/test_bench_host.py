"""Host logic of bench.py, on the CPU: the algorithmic byte counts behind every GB/s
figure, the launch-flag rule that decides which launches may overlap, the traffic
record lookup, the threaded CPU-oracle harness and the reference arm's JSON line."""
from __future__ import annotations

import contextlib
import io
import json

import pytest

import bench
import layer_wise_paged_gb300 as kvl
import workloads

OV, SH, RD = kvl.KVL_LAUNCH_OVERLAP_PREVIOUS, kvl.KVL_LAUNCH_SHARE_SMS, kvl.KVL_LAUNCH_PLAN_READY


def test_llama_layer_bytes_follow_the_kv_size_formula():
    # KV bytes of one layer = 2 (K, V) * T * H_kv * d * 2 bytes (bf16); each op reads
    # its bytes once and writes them once
    spec = workloads.get_spec("llama3_8b_agentic")
    T_hit, T_all = 30720, 30720 + 512
    layer_kv = lambda T: 2 * T * 8 * 128 * 2
    b = bench.op_bytes(spec)
    assert b["slice"] == 2 * layer_kv(T_hit)
    assert b["merge_scatter"] == 2 * layer_kv(T_all)
    # objects carry whole blocks: ceil(T_all / 16) blocks of 16 slots per plane
    nblk = -(-T_all // 16)
    assert b["gather"] == b["scatter_back"] == 2 * 2 * nblk * 16 * 2048
    assert bench.step_bytes(spec) == spec.L * sum(b.values())


@pytest.mark.parametrize("name", ["tiny", "qwen3_32b_long", "latent_batch", "many_small"])
def test_op_bytes_match_the_spec(name):
    spec = workloads.get_spec(name)
    b = bench.op_bytes(spec)
    t_hit, t_all = sum(spec.t_hit), sum(spec.t_hit) + sum(spec.t_miss)
    assert b["slice"] == 2 * t_hit * spec.R
    assert b["merge_scatter"] == 2 * t_all * spec.R
    assert b["gather"] == 2 * spec.P * int(spec.nblk().sum()) * spec.B * spec.Rp


def _flags(op, n, *, ring=8, shared=False, serial=False, K=1, ready=False):
    return [bench.phase_launch_flags(op, i, i * K, ring=ring, n_launches=n,
                                     shared_objects=shared, serial=serial, plan_ready=ready)
            for i in range(n)]


def test_first_launch_of_a_phase_never_overlaps():
    for op in bench.OPS:
        f = _flags(op, 32)
        assert f[0] == SH and not f[0] & OV
        assert all(x == OV for x in f[1:]) or op == "slice"


def test_slice_launches_that_reuse_a_ring_buffer_wait():
    f = _flags("slice", 32, ring=8)
    for i, x in enumerate(f):
        assert (x & OV == 0) == (i % 8 == 0), i
    # several layers per launch: ring is a multiple of K, the check is on first layers
    f = _flags("slice", 8, ring=8, K=4)
    assert [bool(x & OV) for x in f] == [False, True, False, True, False, True, False, True]


def test_shared_object_layer_keeps_gather_and_scatter_back_alone():
    assert _flags("gather", 32, shared=True) == [0] * 32
    assert _flags("scatter_back", 32, shared=True) == [0] * 32
    assert _flags("merge_scatter", 32, shared=True)[1:] == [OV] * 31


def test_serial_and_single_launch_phases_carry_no_flags():
    for op in bench.OPS:
        assert _flags(op, 32, serial=True) == [0] * 32
        assert _flags(op, 1) == [0]


def test_plan_ready_goes_on_every_waiting_launch_but_the_first_after_the_plan():
    # the step's first launch (the slice of layer 0) follows the plan's kernels
    f = _flags("slice", 32, ready=True)
    assert f[0] == SH and all(x & RD for x in f[8::8]) and all(x == OV for x in f[1:8])
    for op in bench.OPS[1:]:
        g = _flags(op, 32, ready=True)
        assert g[0] == SH | RD and g[1:] == [OV] * 31  # an overlapping launch needs no prefetch
    assert _flags("gather", 4, shared=True, ready=True) == [RD] * 4
    assert _flags("merge_scatter", 3, serial=True, ready=True) == [RD] * 3
    assert _flags("slice", 3, serial=True, ready=True) == [0, RD, RD]
    assert _flags("merge_scatter", 3, serial=True) == [0] * 3


@pytest.mark.parametrize("k", [1, 2, 8, 300])
@pytest.mark.parametrize("name", ["many_small", "latent_batch", "llama3_8b_agentic"])
def test_end_to_end_parts_cover_the_requests_in_order(name, k):
    from layer_wise_paged_gb300.shard import request_weights
    spec = workloads.get_spec(name)
    parts = bench.request_parts(spec, k)
    n = spec.n_req
    # the midpoint rule can leave a rank empty only when parts are about as many as
    # requests; empty parts are dropped
    assert 1 <= len(parts) <= min(k, n)
    if k <= 8:
        assert len(parts) == min(k, n)
    # contiguous, non-empty, in order, every request once
    assert parts[0][0] == 0 and parts[-1][1] == n
    assert all(a < z for a, z in parts)
    assert all(parts[i][1] == parts[i + 1][0] for i in range(len(parts) - 1))
    # the midpoint rule's bound: each part within the largest request of an equal share
    w = request_weights(spec.t_hit, spec.t_miss, spec.B)
    share = w.sum() / min(k, n)
    for a, z in parts:
        assert abs(int(w[a:z].sum()) - share) <= int(w.max())


def test_traffic_record_is_read_only_for_the_current_kernel_source():
    h = bench.kernel_source_hash()
    rec = [line.split() for line in (bench.ROOT / "profiles" / "dram_traffic.txt").read_text()
           .splitlines() if line and not line.startswith("#")]
    for kernel, workload, sha, nbytes in rec:
        got = bench.recorded_traffic(kernel, workload)
        assert got == (int(nbytes) if sha == h else None)
    assert bench.recorded_traffic("no_such_kernel", "llama3_8b_agentic") is None


def test_reference_arm_prints_one_json_line():
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2",
                         "--warmup", "3"])
    assert rc == 0
    lines = [x for x in out.getvalue().splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == bench.UNIT and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["higher_is_better"] is True
    # the same scaling label as the GPU arm: the total work does not grow with N
    assert d["scaling"] == "strong"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny"


def test_cpu_baseline_times_the_oracle_on_several_threads():
    spec = workloads.get_spec("tiny")
    cpu = bench.cpu_baseline(spec, budget_s=0.2, threads=2)
    assert cpu["kind"] == "oracle" and cpu["unit"] == bench.UNIT
    assert cpu["value"] > 0 and cpu["single_thread_value"] > 0
    assert 1 <= cpu["cores"] <= 2 and cpu["cores_available"] >= cpu["cores"]


def test_oracle_workers_share_inputs_and_own_their_outputs():
    spec = workloads.get_spec("tiny")
    sample = bench.OracleSample(spec)
    a, b = bench.oracle_workers(sample, 2)
    assert a.hit is b.hit and a.miss is b.miss
    assert a.pool is not b.pool and a.objects is not b.objects
    # every layer done once, whatever the thread count
    nbytes, _, layers = bench.time_oracle([a, b], range(spec.L), float("inf"))
    assert layers == spec.L and nbytes == spec.L * sum(bench.op_bytes(spec).values())
    # each worker's pool holds what one worker alone computes for the same layer
    c = bench.oracle_workers(bench.OracleSample(spec), 1)[0]
    a.run(spec.L - 1)
    c.run(spec.L - 1)
    assert (a.pool == c.pool).all() and (a.objects == c.objects).all()
