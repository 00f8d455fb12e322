"""GPU parity in the benchmark's own launch configuration.

One step exactly as bench.py enqueues it (bench.BenchStep: the plan, then each op over
all layers, successive layers' launches overlapping with the 96 KiB pipelines, the
hit_layer ring, the bench's object layout) on each full-size workload.  Sampled layers
are compared byte for byte with the oracle after every phase; the scatter-back round
trip is checked on every layer.
"""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import pytest
import torch

import workloads
from tests._device import one_layer_problem

pytestmark = pytest.mark.gpu

FULL = ["llama3_8b_agentic", "qwen3_32b_long", "latent_batch", "many_small"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    kvl.lib()


def _equal(got_t, want, what):
    got = got_t.cpu().numpy()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[0]}")


def _fingerprint(region):
    """Two wrapping int64 sums over the region's int32 words (plain and position-mixed):
    equal regions give equal pairs; a changed word changes them unless two changes
    cancel in both sums."""
    w = region.view(torch.int32).to(torch.int64)
    idx = torch.arange(w.numel(), device=w.device, dtype=torch.int64)
    return int(w.sum()), int((w * (idx * 2654435761 + 1)).sum())


@pytest.mark.parametrize("name", FULL)
def test_bench_step_full_size(name):
    import bench
    spec = workloads.get_spec(name)
    one_layer = workloads.footprint_bytes(spec) > 160e9
    need = workloads.footprint_bytes(spec, objects_one_layer=one_layer) / 1e9
    # free to the driver plus free inside torch's cache
    free = (torch.cuda.mem_get_info()[0] + torch.cuda.memory_reserved()
            - torch.cuda.memory_allocated()) / 1e9
    if need + 12 > free:
        pytest.skip(f"{name} needs {need:.0f} GB of device memory, {free:.0f} GB free")
    bs = bench.BenchStep(spec, "cuda")
    assert bs.one_layer == one_layer
    lay, bufs, pool, L = bs.bufs["layout"], bs.bufs, bs.pool, spec.L
    lb = spec.P * spec.n_pool * spec.B * spec.Rp
    region = lambda l: pool[l * lb:(l + 1) * lb]
    sampled = sorted({0, L // 2, L - 1})
    s = torch.cuda.current_stream()
    phases = dict(bs.phases(bs.batch, s))
    # the launch flags are the bench's: overlapping after the first launch of a phase
    assert any(bs.flags("merge_scatter", i, l0) for i, (l0, _) in enumerate(bs.groups))

    bs.batch.plan(stream=s)
    before = {l: region(l).cpu().numpy() for l in sampled}
    dev = SimpleNamespace(hit=bufs["hit"], miss=bufs["miss"], tables=bufs["tables"],
                          src_tables=bufs["src_tables"])
    probs = {l: one_layer_problem(spec, lay, dev, l, before[l]) for l in sampled}

    for launch in phases["slice"]:
        launch()
    torch.cuda.synchronize()
    for l in sampled:
        if l >= L - bs.ring:  # still in the hit_layer ring
            st, want = probs[l][0].slice_layer(0)
            assert st == 0
            _equal(bs.hit_views[l][:want.size], want, f"{name} hit_layer[{l}]")

    for launch in phases["merge_scatter"]:
        launch()
    torch.cuda.synchronize()
    merged_fp = None if one_layer else [_fingerprint(region(l)) for l in range(L)]
    for l in sampled:
        ob, objs, offs, host_pool = probs[l]
        assert ob.merge_scatter(0, host_pool)[0] == 0
        _equal(region(l), host_pool, f"{name} pool layer {l} after merge-scatter")

    for launch in phases["gather"]:
        launch()
    torch.cuda.synchronize()
    for l in sampled:
        ob, objs, offs, host_pool = probs[l]
        assert ob.gather_objects(0, host_pool) == 0
        if one_layer and l != L - 1:
            continue  # the shared object layer holds the last layer's gather
        for q, o in zip(lay.requests, offs):
            nb = spec.P * (-(-(q.t_hit + q.t_miss) // spec.B)) * spec.B * spec.Rp
            a = q.obj_off + l * q.obj_layer_stride
            _equal(bufs["objects"][a:a + nb], objs[o:o + nb], f"{name} objects of layer {l}")

    for launch in phases["scatter_back"]:
        launch()
    torch.cuda.synchronize()
    if not one_layer:
        # gather then scatter-back restores every layer's pool region
        for l in range(L):
            assert _fingerprint(region(l)) == merged_fp[l], f"{name}: round trip, layer {l}"
        for l in sampled:
            _equal(region(l), probs[l][3], f"{name} pool layer {l} after scatter-back")
    else:
        # every layer received the shared objects, i.e. the last layer's blocks
        last_objs = probs[L - 1][1]
        for l in sampled:
            ob, objs, offs, host_pool = probs[l]
            objs[:] = last_objs
            assert ob.scatter_back(0, host_pool) == 0
            _equal(region(l), host_pool, f"{name} pool layer {l} after scatter-back")
    assert bs.batch.status() == (0, 0)
    del bs, bufs, pool, probs, phases, region, dev
    torch.cuda.empty_cache()
