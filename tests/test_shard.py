"""One batch split across ranks (layer_wise_paged_gb300.shard), on the CPU.

Each rank takes a contiguous run of requests (or of layers, when there are fewer
requests than ranks) with its own pool, plan and objects and no data-path exchange.
Checked here without a GPU: the parts cover every request (or layer) exactly once and
every used pool block exactly once; the ranks' byte shares stay within the stated
bound; and, in two gloo ranks on 127.0.0.1, each rank's oracle results on its own part
(inputs cut from the whole batch's) equal the whole batch's oracle results byte for
byte: its pool blocks at their batch-wide ids, its requests' objects, its layers.
"""
from __future__ import annotations

import dataclasses
import os
import socket
from types import SimpleNamespace

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import workloads
from layer_wise_paged_gb300.shard import request_weights, split_batch, split_requests
from tests._host import host_buffers


def _parts(spec, world):
    return [split_batch(spec.t_hit, spec.t_miss, spec.B, spec.L, workloads.block_tables(spec),
                        workloads.source_tables(spec), world, r) for r in range(world)]


@pytest.mark.parametrize("name", ["many_small", "latent_batch"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_request_split_covers_everything_once_and_balances_bytes(name, world):
    spec = workloads.get_spec(name)
    parts = _parts(spec, world)
    reqs = [i for p in parts for i in p.requests]
    assert reqs == list(range(spec.n_req))  # each request once, in order
    ids = np.concatenate([p.pool_ids for p in parts])
    used = workloads.block_tables(spec)
    assert np.array_equal(np.sort(ids), np.sort(used))  # each used block once
    w = request_weights(spec.t_hit, spec.t_miss, spec.B) * spec.L
    total = int(w.sum())
    assert sum(p.weight for p in parts) == total
    for p in parts:
        assert p.kind == "requests" and p.layers == (0, spec.L)
        assert abs(p.weight - total / world) <= int(w.max())  # the stated bound
        # the renumbered tables address the rank's pool and map back to the batch ids
        assert p.tables.min() >= 0 and p.tables.max() < len(p.pool_ids)
        i0, i1 = p.requests[0], p.requests[-1] + 1
        off = np.concatenate([[0], np.cumsum(spec.nblk())])
        assert np.array_equal(p.pool_ids[p.tables], used[off[i0]:off[i1]])


def test_midpoint_rule_is_contiguous_and_exact_on_equal_weights():
    assert list(split_requests([5] * 8, 4)) == [0, 0, 1, 1, 2, 2, 3, 3]
    r = split_requests([1, 100, 1, 1, 1], 2)
    assert list(r) == sorted(r)
    assert list(split_requests([3, 3], 1)) == [0, 0]


def test_fewer_requests_than_ranks_splits_layers():
    spec = workloads.get_spec("qwen3_32b_long")
    parts = _parts(spec, 3)
    assert [p.kind for p in parts] == ["layers"] * 3
    assert [p.layers for p in parts] == [(0, 22), (22, 43), (43, 64)]
    # idle ranks only when there are more ranks than requests and layers
    tiny = workloads.get_spec("tiny")
    assert [p.kind for p in _parts(tiny, 3)] == ["layers", "layers", "idle"]


def test_part_spec_allocates_the_part():
    spec = workloads.get_spec("many_small")
    p = _parts(spec, 4)[2]
    ps = workloads.part_spec(spec, p)
    assert ps.n_req == len(p.requests) and ps.n_pool == len(p.pool_ids)
    assert np.array_equal(workloads.block_tables(ps), p.tables)
    assert int(ps.nblk().sum()) == len(p.pool_ids)  # injective tables: no headroom needed


# ---- two gloo ranks: the parts' oracle results equal the whole batch's ----------

SPEC = workloads.custom_spec(L=3, P=2, B=4, Rp=32, t_hit=[13, 0, 7, 30, 2, 9],
                             t_miss=[3, 5, 0, 6, 1, 4], table="perm", source="permuted",
                             seed=77)
SPEC_1REQ = workloads.custom_spec(L=5, P=2, B=4, Rp=32, t_hit=[21], t_miss=[6],
                                  table="perm", source="permuted", seed=78)


def _geom(spec):
    return SimpleNamespace(L=spec.L, P=spec.P, B=spec.B, Rp=spec.Rp, n_pool=spec.n_pool)


def _run_all(spec, hb):
    """Oracle slice, merge-scatter and gather of every layer; returns (hit_layers, pool,
    objects)."""
    ob = oracle.Batch(_geom(spec), hb.layout.requests, hb.hit, hb.miss, hb.objects, hb.tables,
                      hb.src_tables)
    hits = []
    for l in range(spec.L):
        st, h = ob.slice_layer(l)
        assert st == 0
        hits.append(h)
        assert ob.merge_scatter(l, hb.pool)[0] == 0
        assert ob.gather_objects(l, hb.pool) == 0
    return hits, hb.pool, hb.objects


def _part_inputs(spec, hb, part):
    """The rank's host inputs, cut from the whole batch's: its requests' full blocks,
    miss rows and tables (request split), or its layers of every row (layer split)."""
    ps = workloads.part_spec(spec, part)
    lay = workloads.layout(ps)
    R, L = spec.R, spec.L
    if part.kind == "requests":
        i0, i1 = part.requests[0], part.requests[-1] + 1
        rq = hb.layout.requests
        end_hit = rq[i1].hit_off if i1 < spec.n_req else hb.layout.hit_bytes
        end_miss = rq[i1].miss_off if i1 < spec.n_req else hb.layout.miss_bytes
        hit = hb.hit[rq[i0].hit_off:end_hit].copy()
        miss = hb.miss[rq[i0].miss_off:end_miss].copy()
    else:
        l0, l1 = part.layers
        rows = hb.layout.hit_bytes // (L * R)
        hit = hb.hit[:rows * L * R].reshape(rows, L, R)[:, l0:l1].reshape(-1).copy()
        # miss rows are layer-major per request: [L, T_miss, R]
        parts = [hb.miss[q.miss_off:q.miss_off + L * q.t_miss * R].reshape(L, q.t_miss * R)[l0:l1]
                 .reshape(-1) for q in hb.layout.requests]
        miss = np.concatenate(parts) if parts else np.zeros(0, np.uint8)
    assert hit.size == lay.hit_bytes and miss.size == lay.miss_bytes
    pad = lambda a: np.concatenate([a, np.zeros(64, np.uint8)])
    return ps, SimpleNamespace(layout=lay, hit=pad(hit), miss=pad(miss),
                               pool=np.full(lay.pool_bytes + 64, workloads.SENTINEL, np.uint8),
                               objects=np.full(lay.obj_bytes + 64, workloads.SENTINEL, np.uint8),
                               tables=part.tables, src_tables=part.src_tables)


def _rank_main(rank, world, port, which, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo")
    spec = SPEC if which == "requests" else SPEC_1REQ
    hb = host_buffers(spec)  # every rank draws the whole batch's inputs from the same seed
    whole = host_buffers(spec)
    want_hits, want_pool, want_obj = _run_all(spec, whole)
    part = split_batch(spec.t_hit, spec.t_miss, spec.B, spec.L, hb.tables, hb.src_tables,
                       world, rank)
    ps, pin = _part_inputs(spec, hb, part)
    hits, pool, objs = _run_all(ps, pin)
    # compare this rank's results with the whole batch's, at their batch-wide places
    P, N, B, Rp, L = spec.P, spec.n_pool, spec.B, spec.Rp, spec.L
    wpool = want_pool[:L * P * N * B * Rp].reshape(L, P, N, B * Rp)
    l0, l1 = part.layers
    gpool = pool[:(l1 - l0) * P * len(part.pool_ids) * B * Rp].reshape(l1 - l0, P, len(part.pool_ids), B * Rp)
    ok = np.array_equal(gpool, wpool[l0:l1][:, :, part.pool_ids])
    wl = whole.layout
    for k, i in enumerate(part.requests):
        q, qw = pin.layout.requests[k], wl.requests[i]
        nb = -(-(q.t_hit + q.t_miss) // B)
        for l in range(l1 - l0):
            for p in range(P):
                a = q.obj_off + l * q.obj_layer_stride + p * q.obj_plane_stride
                b = qw.obj_off + (l0 + l) * qw.obj_layer_stride + p * qw.obj_plane_stride
                ok &= np.array_equal(objs[a:a + nb * B * Rp], want_obj[b:b + nb * B * Rp])
    hit_off = np.concatenate([[0], np.cumsum(spec.t_hit)]) * spec.R
    for l in range(l1 - l0):
        want = np.concatenate([want_hits[l0 + l][hit_off[i]:hit_off[i + 1]] for i in part.requests])
        ok &= np.array_equal(hits[l], want)
    # every rank must agree that all of the batch was covered exactly once
    cover = [None] * world
    dist.all_gather_object(cover, (list(part.requests), part.layers, part.pool_ids.tolist()))
    out.put((rank, bool(ok), cover))
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("which", ["requests", "layers"])
def test_two_gloo_ranks_reproduce_the_whole_batch(which):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, which, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, ok, cover = q.get(timeout=180)
        res[r] = (ok, cover)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(ok for ok, _ in res.values()), res
    cover = res[0][1]
    assert cover == res[1][1]
    spec = SPEC if which == "requests" else SPEC_1REQ
    if which == "requests":
        assert sorted(i for c in cover for i in c[0]) == list(range(spec.n_req))
        ids = sorted(i for c in cover for i in c[2])
        assert ids == sorted(workloads.block_tables(spec).tolist())
    else:
        layers = sorted(l for c in cover for l in range(*c[1]))
        assert layers == list(range(spec.L))
