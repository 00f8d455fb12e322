"""One batch split across GPUs, one process per GPU, with no data-path exchange.

The reshuffle of one request touches only that request's rows, blocks and objects,
and the reshuffle of one layer only that layer's (Tutti 阅读笔记, 伪代码 1: retrieve_layer
works per layer on a request's own block ids).  So a batch splits into independent
parts: each rank takes a contiguous run of requests (or, when there are fewer
requests than ranks, a contiguous run of layers of every request), keeps its own pool,
plan and objects, and exchanges nothing with the others.  A rank's pool holds only the
pool blocks its requests use, renumbered in increasing order of their batch-wide ids:
local block k is batch block ``pool_ids[k]``.

Host logic only: integer partitioning of counts and renumbering of block tables.  It
moves no KV bytes and does none of the reshuffle; each rank then calls the library
on its part exactly as a one-GPU caller does.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Part:
    """What one rank of `world` processes.

    kind      "requests" (a run of requests, every layer), "layers" (every request, a
              run of layers) or "idle" (nothing: more ranks than requests and layers)
    requests  indices of the batch's requests the rank processes, in order
    layers    (l0, l1): the rank processes layers l0 <= l < l1
    pool_ids  batch-wide pool block ids held by the rank's own pool, increasing;
              the rank's block k is batch block pool_ids[k]
    tables    the rank's packed block tables (int32), renumbered into its own pool
    src_tables  the rank's packed full-block tables (None if the batch has none);
              full-block ids index each request's own source, so they are not renumbered
    weight    the rank's share of the step's algorithmic bytes, in token rows of one layer
    """
    rank: int
    world: int
    kind: str
    requests: tuple
    layers: tuple
    pool_ids: np.ndarray
    tables: np.ndarray
    src_tables: np.ndarray | None
    weight: int


def request_weights(t_hit, t_miss, B: int) -> np.ndarray:
    """Each request's algorithmic bytes in one step, in token rows of one layer: the
    slice moves its hit rows, the merge-scatter its hit and miss rows, gather and
    scatter-back its whole blocks, each read once and written once."""
    th = np.asarray(t_hit, np.int64)
    ta = th + np.asarray(t_miss, np.int64)
    nblk = -(-ta // B)
    return 2 * th + 2 * ta + 4 * nblk * B


def split_requests(weights, world: int) -> np.ndarray:
    """Rank of each request: contiguous runs, balanced by weight.  A request goes to
    the rank whose share [r/world, (r+1)/world) of the total holds the midpoint of its
    own weight; so each rank's weight differs from total/world by at most the largest
    single weight."""
    w = np.asarray(weights, np.int64)
    total = int(w.sum())
    if world <= 1 or w.size == 0 or total == 0:
        return np.zeros(w.size, np.int64)
    before = np.concatenate([[0], np.cumsum(w)[:-1]])
    mid2 = 2 * before + w  # twice the midpoint, in integers
    return np.minimum(world - 1, (world * mid2) // (2 * total))


def split_layers(L: int, world: int, rank: int) -> tuple:
    """Contiguous layer run of `rank`: L // world layers each, one more for the first
    L % world ranks."""
    base, extra = divmod(L, world)
    l0 = rank * base + min(rank, extra)
    return (l0, l0 + base + (1 if rank < extra else 0))


def split_batch(t_hit, t_miss, B: int, L: int, tables, src_tables, world: int, rank: int) -> Part:
    """Rank `rank`'s part of a batch (see the module docstring).

    t_hit, t_miss: per-request token counts; B: tokens per block; L: layers;
    tables: the batch's packed block tables (int32, request order); src_tables: the
    packed full-block tables (ceil(T_hit / B) entries per request) or None.
    """
    t_hit = np.asarray(t_hit, np.int64)
    t_miss = np.asarray(t_miss, np.int64)
    tables = np.asarray(tables, np.int32)
    n = t_hit.size
    nblk = -(-(t_hit + t_miss) // B)
    blk_off = np.concatenate([[0], np.cumsum(nblk)])
    nsrc = -(-t_hit // B)
    src_off = np.concatenate([[0], np.cumsum(nsrc)])
    w = request_weights(t_hit, t_miss, B)
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if n >= world:
        ranks = split_requests(w, world)
        mine = np.nonzero(ranks == rank)[0]
        if mine.size == 0:
            return _idle(rank, world, src_tables)
        i0, i1 = int(mine[0]), int(mine[-1]) + 1
        own = tables[blk_off[i0]:blk_off[i1]]
        pool_ids = np.unique(own).astype(np.int64)
        local = np.searchsorted(pool_ids, own).astype(np.int32)
        src = None if src_tables is None else np.asarray(src_tables, np.int32)[src_off[i0]:src_off[i1]].copy()
        return Part(rank, world, "requests", tuple(range(i0, i1)), (0, L), pool_ids, local, src,
                    int(w[i0:i1].sum()) * L)
    l0, l1 = split_layers(L, world, rank)
    if l1 <= l0:
        return _idle(rank, world, src_tables)
    own = tables[:blk_off[n]]
    pool_ids = np.unique(own).astype(np.int64)
    local = np.searchsorted(pool_ids, own).astype(np.int32)
    src = None if src_tables is None else np.asarray(src_tables, np.int32).copy()
    return Part(rank, world, "layers", tuple(range(n)), (l0, l1), pool_ids, local, src,
                int(w.sum()) * (l1 - l0))


def _idle(rank, world, src_tables) -> Part:
    return Part(rank, world, "idle", (), (0, 0), np.zeros(0, np.int64), np.zeros(0, np.int32),
                None if src_tables is None else np.zeros(0, np.int32), 0)
