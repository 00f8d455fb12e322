"""Host-side (numpy) buffers for tests: payloads, tagged payloads, guards.

Builds the same packed buffers the workloads module lays out, in numpy, so the
oracle can run on them; and the tag payload the pin tests decode.
"""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np

import workloads

GUARD = 64  # bytes of sentinel after every output buffer; an overrun shows up there


def geom_of(spec):
    return SimpleNamespace(L=spec.L, P=spec.P, B=spec.B, Rp=spec.Rp, n_pool=spec.n_pool)


def _random_bytes(n, seed):
    return np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8)


def host_buffers(spec, *, payload="bytes", objects_one_layer=False, seed=7):
    """Packed numpy buffers for `spec`: hit, miss (payload), pool, objects (sentinel)."""
    lay = workloads.layout(spec, objects_one_layer=objects_one_layer)
    hit = _random_bytes(lay.hit_bytes + GUARD, seed)
    miss = _random_bytes(lay.miss_bytes + GUARD, seed + 1)
    pool = np.full(lay.pool_bytes + GUARD, workloads.SENTINEL, np.uint8)
    objects = np.full(lay.obj_bytes + GUARD, workloads.SENTINEL, np.uint8)
    tables = workloads.block_tables(spec)
    src_tables = workloads.source_tables(spec)
    if payload == "tags":
        write_tags(spec, lay, hit, miss, src_tables)
    return SimpleNamespace(spec=spec, layout=lay, hit=hit, miss=miss, pool=pool,
                           objects=objects, tables=tables, src_tables=src_tables)


def tag(r, t, l, p, kind):
    """16-byte tag of (request, token index in complete_layer, layer, plane, hit/miss)."""
    return np.array([r, t, l, p + 16 * kind], dtype=np.int32)


def write_tags(spec, lay, hit, miss, src_tables):
    """Write a tag into every Rp-byte plane row of every hit and miss token.

    Hit token t of request r, layer l, plane p carries tag(r, t, l, p, 0); miss token m
    carries tag(r, T_hit + m, l, p, 1), i.e. its position in complete_layer.  The
    16-byte tag is repeated across the row.
    """
    assert spec.Rp % 16 == 0
    reps = spec.Rp // 16
    for r, q in enumerate(lay.requests):
        for t in range(q.t_hit):
            j, s = divmod(t, spec.B)
            blk = j if q.src_table_off < 0 else int(src_tables[q.src_table_off + j])
            for l in range(spec.L):
                for p in range(spec.P):
                    off = (q.hit_off + blk * q.hit_block_stride + s * q.hit_token_stride
                           + l * q.hit_layer_stride + p * spec.Rp)
                    hit[off:off + spec.Rp] = np.tile(tag(r, t, l, p, 0), reps).view(np.uint8)
        for m in range(q.t_miss):
            for l in range(spec.L):
                for p in range(spec.P):
                    off = (q.miss_off + m * q.miss_token_stride + l * q.miss_layer_stride
                           + p * spec.Rp)
                    miss[off:off + spec.Rp] = np.tile(tag(r, q.t_hit + m, l, p, 1),
                                                      reps).view(np.uint8)


def decode_rows(buf_u8, Rp):
    """View a buffer of Rp-byte rows as tags; None for rows that are not one tag repeated."""
    rows = np.ascontiguousarray(buf_u8).view(np.int32).reshape(-1, Rp // 16, 4)
    first = rows[:, :1, :]
    uniform = np.all(rows == first, axis=(1, 2))
    return rows[:, 0, :], uniform
