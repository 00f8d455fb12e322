"""GPU parity in the benchmark's own launch configuration, on every layer.

One step exactly as bench.py enqueues it (bench.BenchStep: the plan, then each op over
all layers, successive layers' launches overlapping with the 96 KiB pipelines, the
hit_layer ring, the bench's object layout) on each full-size workload.  After every
phase, every layer is compared byte for byte with the oracle, each op's oracle applied
to the layer's inputs (the pool it reads having been checked already).  A phase is
paused only where the bench's launch rule already makes a launch wait for the one
before it (a slice launch that reuses a hit_layer ring buffer; every gather when all
layers share one object layer), so each layer's output can be read before the next
launch overwrites it.

The end-to-end steps of bench.EndToEnd (inputs uploaded from pinned host memory, or
read there in place by the slice and merge-scatter; objects read back to pinned host
memory) are compared with the oracle on sampled layers.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import workloads
from tests._device import one_layer_problem

pytestmark = pytest.mark.gpu

FULL = ["llama3_8b_agentic", "qwen3_32b_long", "latent_batch", "many_small"]
THREADS = 4  # layers checked at once (the oracle's C calls release the GIL)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    kvl.lib()


def _equal(got_t, want, what):
    got = got_t.cpu().numpy() if isinstance(got_t, torch.Tensor) else got_t
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[0]}")


def _each(fn, items, threads=THREADS):
    with ThreadPoolExecutor(threads) as ex:
        for f in [ex.submit(fn, x) for x in items]:
            f.result()


def _free_gb():
    return (torch.cuda.mem_get_info()[0] + torch.cuda.memory_reserved()
            - torch.cuda.memory_allocated()) / 1e9


class Layers:
    """The oracle of one layer at a time, over the device inputs of a full workload."""

    def __init__(self, spec, bs):
        self.spec, self.bs = spec, bs
        b = bs.bufs
        self.lay = b["layout"]
        self.dev = SimpleNamespace(hit=b["hit"], miss=b["miss"], tables=b["tables"],
                                   src_tables=b["src_tables"])
        self.lb = spec.P * spec.n_pool * spec.B * spec.Rp

    def region(self, l):
        return self.bs.pool[l * self.lb:(l + 1) * self.lb]

    def problem(self, l, pool_before=None):
        if pool_before is None:
            pool_before = np.full(self.lb, workloads.SENTINEL, np.uint8)
        return one_layer_problem(self.spec, self.lay, self.dev, l, pool_before)

    def objects_of(self, l):
        """(device bytes, per-request (offset, size)) of layer l's objects."""
        spec, out = self.spec, []
        for q in self.lay.requests:
            nb = spec.P * (-(-(q.t_hit + q.t_miss) // spec.B)) * spec.B * spec.Rp
            out.append((q.obj_off + l * q.obj_layer_stride, nb))
        return out


@pytest.mark.parametrize("name,serial", [(n, False) for n in FULL] + [("llama3_8b_agentic", True)],
                         ids=FULL + ["llama3_8b_agentic-serial"])
def test_bench_step_full_size_every_layer(name, serial):
    """serial: every launch alone, each after the first prefetching before its wait
    (KVL_LAUNCH_PLAN_READY), as the bench's serial step runs them."""
    import bench
    import layer_wise_paged_gb300 as kvl
    spec = workloads.get_spec(name)
    one_layer = workloads.footprint_bytes(spec) > 160e9
    need = workloads.footprint_bytes(spec, objects_one_layer=one_layer) / 1e9
    if need + 12 + 4 * 3 > _free_gb():
        pytest.skip(f"{name} needs {need:.0f} GB of device memory, {_free_gb():.0f} GB free")
    bs = bench.BenchStep(spec, "cuda", serial=serial)
    assert bs.one_layer == one_layer
    L, ring = spec.L, bs.ring
    chk = Layers(spec, bs)
    s = torch.cuda.current_stream()
    phases = dict(bs.phases(bs.batch, s))
    flags = {op: [bs.flags(op, i, l0) for i, (l0, _) in enumerate(bs.groups)] for op in bench.OPS}
    # the launch flags are the bench's: overlapping after the first launch of a phase
    # (serial: none overlapping, every one but the step's first prefetching)
    if serial:
        ov = kvl.KVL_LAUNCH_OVERLAP_PREVIOUS
        assert not any(f & ov for fl in flags.values() for f in fl)
        assert all(f & kvl.KVL_LAUNCH_PLAN_READY for f in flags["merge_scatter"])
    else:
        assert any(flags["merge_scatter"])
    bs.batch.plan(stream=s)

    # slice: a launch whose first layer reuses a ring buffer waits for the one before it,
    # so the phase pauses there and the ring's layers are checked before being rewritten
    def check_slice(l):
        st, want = chk.problem(l)[0].slice_layer(0)
        assert st == 0
        _equal(bs.hit_views[l][:want.size], want, f"{name} hit_layer[{l}]")

    done = 0
    for i, launch in enumerate(phases["slice"]):
        if i and bs.groups[i][0] % ring == 0:
            assert not flags["slice"][i] & kvl.KVL_LAUNCH_OVERLAP_PREVIOUS
            torch.cuda.synchronize()
            _each(check_slice, range(done, bs.groups[i][0]))
            done = bs.groups[i][0]
        launch()
    torch.cuda.synchronize()
    _each(check_slice, range(done, L))

    # merge-scatter: every layer's pool region against the oracle's slice, concatenate
    # and scatter of that layer into a sentinel region
    for launch in phases["merge_scatter"]:
        launch()
    torch.cuda.synchronize()

    def check_merge(l):
        ob, _, _, host_pool = chk.problem(l)
        assert ob.merge_scatter(0, host_pool)[0] == 0
        _equal(chk.region(l), host_pool, f"{name} pool layer {l} after merge-scatter")
    _each(check_merge, range(L))

    # gather: each layer's objects against the oracle's gather of that (checked) region
    def check_gather(l):
        ob, objs, offs, host_pool = chk.problem(l, chk.region(l).cpu().numpy())
        assert ob.gather_objects(0, host_pool) == 0
        for (a, nb), o in zip(chk.objects_of(l), offs):
            _equal(bs.bufs["objects"][a:a + nb], objs[o:o + nb], f"{name} objects of layer {l}")

    if one_layer:
        # every gather runs alone (one shared object layer): check each before the next
        assert not any(f & kvl.KVL_LAUNCH_OVERLAP_PREVIOUS for f in flags["gather"])
        for i, launch in enumerate(phases["gather"]):
            launch()
            torch.cuda.synchronize()
            check_gather(bs.groups[i][0])
    else:
        for launch in phases["gather"]:
            launch()
        torch.cuda.synchronize()
        _each(check_gather, range(L))

    # scatter-back: every layer's region against the oracle's scatter-back of the
    # objects that layer reads (its own, or the shared layer's: the last layer's)
    if one_layer:
        last = chk.problem(L - 1, chk.region(L - 1).cpu().numpy())
        assert last[0].gather_objects(0, last[3]) == 0
        shared = last[1]
    for launch in phases["scatter_back"]:
        launch()
    torch.cuda.synchronize()

    def check_scatter_back(l):
        # the region before scatter-back equals the oracle's merge-scatter result
        ob, objs, offs, host_pool = chk.problem(l)
        assert ob.merge_scatter(0, host_pool)[0] == 0
        if one_layer:
            objs[:] = shared
        else:
            assert ob.gather_objects(0, host_pool) == 0
        assert ob.scatter_back(0, host_pool) == 0
        _equal(chk.region(l), host_pool, f"{name} pool layer {l} after scatter-back")
    _each(check_scatter_back, range(L))
    assert bs.batch.status() == (0, 0)
    del bs, phases, chk
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama3_8b_agentic", "many_small"])
@pytest.mark.parametrize("in_place", [False, True], ids=["staged", "in_place"])
def test_end_to_end_step_full_size(name, in_place):
    """One end-to-end step as bench.py times it: the inputs uploaded from pinned host
    memory (or read there in place by the slice and merge-scatter), the objects read
    back to pinned host memory layer by layer (through a ring of device object slots
    when all layers share one object layer; the 256-request batch in byte-balanced parts
    of its requests, one input set; the Llama turn alternating two input sets).  Sampled
    layers of hit_layer, the pool and the objects read back are compared with the
    oracle."""
    import bench
    spec = workloads.get_spec(name)
    one_layer = workloads.footprint_bytes(spec) > 160e9
    need = workloads.footprint_bytes(spec, objects_one_layer=one_layer) / 1e9
    if need + 12 + 3 * 3 > _free_gb():
        pytest.skip(f"{name} needs {need:.0f} GB of device memory, {_free_gb():.0f} GB free")
    bs = bench.BenchStep(spec, "cuda")
    try:
        ee = bench.EndToEnd(bs, torch.device("cuda"))
    except MemoryError as exc:
        pytest.skip(str(exc))
    L = spec.L
    chk = Layers(spec, bs)
    # the device inputs are cleared: what the step reads must come from the host
    if not in_place:
        bs.bufs["hit"].zero_()
        bs.bufs["miss"].zero_()
    ee.run(1, in_place)
    assert ee.status_ok()
    if not in_place:  # the uploads restored the inputs the oracle reads
        assert np.array_equal(bs.bufs["hit"][:1 << 20].cpu().numpy(), ee.h_hit.np[:1 << 20])
    sampled = sorted({L - bs.ring, L - 2, L - 1})

    def check(l):
        ob, objs, offs, host_pool = chk.problem(l)
        st, want = ob.slice_layer(0)
        assert st == 0
        _equal(bs.hit_views[l][:want.size], want, f"{name} hit_layer[{l}]")
        assert ob.merge_scatter(0, host_pool)[0] == 0
        assert ob.gather_objects(0, host_pool) == 0
        # objects read back: every layer's with an object buffer of all layers; the last
        # two layers' in the two host slots of a shared object layer
        if not one_layer or l >= L - 2:
            host = ee.t_obj[l % 2 if one_layer else 0].numpy()
            for (a, nb), o in zip(chk.objects_of(l), offs):
                _equal(host[a:a + nb], objs[o:o + nb], f"{name} objects of layer {l} on the host")
    _each(check, sampled, threads=3)
    # after scatter-back the pool's layers hold what the oracle's scatter-back gives: a
    # layer's own objects, or with a shared object layer those of the last layer
    # gathered into the ring slot it reads (slot l mod ring)
    def objects_of_layer(j):
        ob, objs, offs, host_pool = chk.problem(j)
        assert ob.merge_scatter(0, host_pool)[0] == 0
        assert ob.gather_objects(0, host_pool) == 0
        return objs

    assert ee.ring == (4 if one_layer else ee.n_sets)
    assert len(ee.parts) == (bench.E2E_PARTS if ee.n_sets == 1 else 1)
    for l in sampled:
        ob, objs, offs, host_pool = chk.problem(l)
        assert ob.merge_scatter(0, host_pool)[0] == 0
        if one_layer:
            objs[:] = objects_of_layer(max(j for j in range(L) if j % ee.ring == l % ee.ring))
        else:
            assert ob.gather_objects(0, host_pool) == 0
        assert ob.scatter_back(0, host_pool) == 0
        _equal(chk.region(l), host_pool, f"{name} pool layer {l} after the end-to-end step")
    ee.close()
    del ee, bs, chk
    torch.cuda.empty_cache()
