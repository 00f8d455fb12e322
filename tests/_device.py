"""Device-side helpers for the GPU tests: copy host inputs to the GPU, build a Batch,
and cut one layer out of a full-size device problem so the oracle can check it."""
from __future__ import annotations

import dataclasses
from types import SimpleNamespace

import numpy as np
import torch

import oracle
import workloads
from layer_wise_paged_gb300.batch import MappedHost
from tests._host import GUARD


def mapped_copy(a: np.ndarray):
    m = MappedHost(a.nbytes)
    m.np[:a.nbytes] = a.view(np.uint8).reshape(-1)
    return m


def to_dev(a: np.ndarray | None):
    if a is None:
        return None
    if a.size == 0:
        a = np.zeros(1, a.dtype)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def device_batch(spec, hb):
    """A GPU Batch over device copies of the host buffers `hb` (same bytes)."""
    from layer_wise_paged_gb300.batch import Batch
    d = SimpleNamespace(hit=to_dev(hb.hit), miss=to_dev(hb.miss), pool=to_dev(hb.pool),
                        objects=to_dev(hb.objects), tables=to_dev(hb.tables),
                        src_tables=to_dev(hb.src_tables))
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    b = Batch(g, hb.layout.requests, d.hit, d.miss, d.objects, d.tables, d.src_tables)
    return b, d


def sentinel_dev(nbytes):
    return torch.full((int(nbytes) + GUARD,), workloads.SENTINEL, dtype=torch.uint8, device="cuda")


def one_layer_problem(spec, lay, dev, layer, pool_before):
    """Host inputs of layer `layer` only, for the oracle (geometry with L = 1).

    dev: the device buffers (hit, miss, tables, src_tables) of the full problem.
    pool_before: numpy bytes of the pool's layer region before the layer's calls.
    Returns (oracle.Batch over host arrays, host objects buffer, per-request object
    offsets in it).
    """
    L, R, B = spec.L, spec.R, spec.B
    # hit rows of this layer: every source layout here has token stride L*R and layer
    # stride R, so the packed buffer viewed as [rows, L, R] gives the layer as [:, l].
    rows = lay.hit_bytes // (L * R)
    hit_l = dev.hit[:rows * L * R].view(rows, L, R)[:, layer, :].contiguous().cpu().numpy().reshape(-1)
    # miss rows of this layer, request by request, packed
    parts, miss_off, off = [], [], 0
    for q in lay.requests:
        miss_off.append(off)
        if q.t_miss:
            a = q.miss_off + layer * q.miss_layer_stride
            if q.miss_token_stride == R:
                t = dev.miss[a:a + q.t_miss * R]
            else:
                t = dev.miss[a:a + (q.t_miss - 1) * q.miss_token_stride + R].as_strided(
                    (q.t_miss, R), (q.miss_token_stride, 1))
            parts.append(t.contiguous().cpu().numpy().reshape(-1))
            off += q.t_miss * R
    miss_l = np.concatenate(parts) if parts else np.zeros(16, np.uint8)
    reqs, obj_off = [], 0
    for r, q in enumerate(lay.requests):
        nblk = -(-(q.t_hit + q.t_miss) // B)
        reqs.append(dataclasses.replace(
            q, hit_off=q.hit_off // L, hit_block_stride=q.hit_block_stride // L,
            hit_token_stride=q.hit_token_stride // L, hit_layer_stride=0,
            miss_off=miss_off[r], miss_token_stride=R, miss_layer_stride=0,
            obj_off=obj_off, obj_layer_stride=0, obj_plane_stride=nblk * B * spec.Rp,
            obj_block_stride=B * spec.Rp))
        obj_off += spec.P * nblk * B * spec.Rp
    objects = np.full(obj_off + GUARD, workloads.SENTINEL, np.uint8)
    g1 = SimpleNamespace(L=1, P=spec.P, B=B, Rp=spec.Rp, n_pool=spec.n_pool)
    tables = dev.tables.cpu().numpy()
    src_tables = None if dev.src_tables is None else dev.src_tables.cpu().numpy()
    ob = oracle.Batch(g1, reqs, hit_l, miss_l, objects, tables, src_tables)
    pool = np.ascontiguousarray(pool_before).copy()
    return ob, objects, [q.obj_off for q in reqs], pool
