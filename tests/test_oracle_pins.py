"""Pins of the CPU oracle to what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself:
* the block and object counts the pages print (Tutti eqs. (3)(4)(14)(15), golden file);
* the KV size of Tutti eq. (1);
* tagged payloads: every output row is decoded back to (request, token, layer, plane,
  hit/miss), which fixes hit-before-miss (DualPath concatenate_tokens) and the token,
  layer and KV-head order the full-block -> layer-block change must keep;
* special cases that reduce to numpy slicing and reshapes (identity tables);
* round trips (scatter-back after gather restores the pool);
* a pure-Python brute force on tiny inputs;
* the plan's prefix sums against numpy's cumsum and its planted errors.
"""
from __future__ import annotations

from pathlib import Path

import numpy as np
import pytest

import oracle
import workloads
from tests._host import decode_rows, geom_of, host_buffers, tag

SENT = workloads.SENTINEL
GOLDEN = Path(__file__).resolve().parent / "golden"

pytestmark = pytest.mark.filterwarnings("ignore")


def batch_of(hb, lib=None):
    return oracle.Batch(geom_of(hb.spec), hb.layout.requests, hb.hit, hb.miss, hb.objects,
                        hb.tables, hb.src_tables, lib=lib)


def _cumsum0(x):
    return np.concatenate([[0], np.cumsum(np.asarray(x, np.int64))])


# --------------------------------------------------------------------------
# Counts the pages print
# --------------------------------------------------------------------------

def golden_counts():
    rows = []
    for line in (GOLDEN / "tutti_counts.txt").read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            L, B, T, blocks, objects, per_layer = line.split()
            rows.append((int(L), int(B), int(T), int(blocks), int(objects),
                         None if per_layer == "-" else int(per_layer)))
    return rows


@pytest.mark.parametrize("row", golden_counts(), ids=lambda r: f"L{r[0]}_B{r[1]}_T{r[2]}")
@pytest.mark.parametrize("hit_frac", [1.0, 0.75])
def test_block_and_object_counts_match_tutti(row, hit_frac, lib=None):
    """ceil(T/B) blocks and 2*L*blocks objects (Tutti eqs. (3)(4), (14)(15))."""
    L, B, T, blocks, objects, per_layer = row
    t_hit = int(T * hit_frac)
    # 1-byte planes: the counts do not depend on the row size, and this keeps it small.
    spec = workloads.custom_spec(L=L, P=2, B=B, Rp=1, t_hit=[t_hit], t_miss=[T - t_hit],
                                 n_pool=blocks, table="identity")
    hb = host_buffers(spec)
    hb.pool[:hb.layout.pool_bytes] = 0
    b = batch_of(hb, lib)
    plan = b.plan()
    assert plan["status"] == oracle.OK
    assert plan["n_items"] == blocks
    obj_bytes = B * spec.Rp
    for layer in range(L):
        assert b.gather_objects(layer, hb.pool) == oracle.OK
        if layer == 0 and per_layer is not None:
            written0 = hb.objects[:hb.layout.obj_bytes].reshape(-1, obj_bytes)
            assert int(np.all(written0 == 0, axis=1).sum()) == per_layer
    objs = hb.objects[:hb.layout.obj_bytes].reshape(-1, obj_bytes)
    assert int(np.all(objs == 0, axis=1).sum()) == objects
    assert np.all(hb.objects[hb.layout.obj_bytes:] == SENT)


def test_object_bytes_equal_tutti_eq1(lib=None):
    """Sum of object bytes over all layers = 2*L*T*H*d*dtype_bytes when B divides T."""
    L, H, d, s, T, B = 3, 2, 4, 2, 96, 16
    spec = workloads.custom_spec(L=L, P=2, B=B, Rp=H * d * s, t_hit=[64], t_miss=[T - 64],
                                 table="perm")
    hb = host_buffers(spec)
    hb.pool[:hb.layout.pool_bytes] = 0
    b = batch_of(hb, lib)
    for layer in range(L):
        assert b.gather_objects(layer, hb.pool) == oracle.OK
    assert int((hb.objects == 0).sum()) == 2 * L * T * H * d * s
    assert np.all(hb.objects[hb.layout.obj_bytes:] == SENT)


# --------------------------------------------------------------------------
# Tagged payloads: order and placement
# --------------------------------------------------------------------------

RAGGED = dict(t_hit=[10, 0, 7, 8, 0, 3], t_miss=[3, 5, 0, 1, 0, 0])


def tagged_spec(source="permuted", miss_order="layer", P=2, table="perm"):
    return workloads.custom_spec(L=3, P=P, B=4, Rp=32, **RAGGED, table=table, source=source,
                                 miss_order=miss_order, seed=11)


def expected_pool_tags(spec, layer):
    """{(p, block, slot): tag} of every pool row a merge-scatter of `layer` writes."""
    tables = workloads.block_tables(spec)
    out, tab0 = {}, 0
    for r, (th, tm) in enumerate(zip(spec.t_hit, spec.t_miss)):
        for t in range(th + tm):
            blk = int(tables[tab0 + t // spec.B])
            for p in range(spec.P):
                out[(p, blk, t % spec.B)] = tag(r, t, layer, p, int(t >= th))
        tab0 += -(-(th + tm) // spec.B)
    return out


def check_pool(spec, pool, layers_done):
    N, B, P, L = spec.n_pool, spec.B, spec.P, spec.L
    tags, uniform = decode_rows(pool[:L * P * N * B * spec.Rp], spec.Rp)
    tags = tags.reshape(L, P, N, B, 4)
    sent_row = np.frombuffer(bytes([SENT]) * 16, np.int32)
    for l in range(L):
        exp = expected_pool_tags(spec, l) if l in layers_done else {}
        for p in range(P):
            for blk in range(N):
                for s in range(B):
                    got = tags[l, p, blk, s]
                    want = exp.get((p, blk, s))
                    if want is None:
                        assert np.array_equal(got, sent_row), (l, p, blk, s, got)
                    else:
                        assert np.array_equal(got, want), (l, p, blk, s, got, want)
    assert np.all(uniform)
    assert np.all(pool[L * P * N * B * spec.Rp:] == SENT)


@pytest.mark.parametrize("source", ["contiguous", "permuted"])
@pytest.mark.parametrize("miss_order", ["layer", "token"])
def test_merge_scatter_places_hit_then_miss_tokens(source, miss_order, lib=None):
    spec = tagged_spec(source, miss_order)
    hb = host_buffers(spec, payload="tags")
    b = batch_of(hb, lib)
    assert b.plan()["status"] == oracle.OK
    done = set()
    for layer in (2, 0, 1):
        st, _ = b.merge_scatter(layer, hb.pool)
        assert st == oracle.OK
        done.add(layer)
        check_pool(spec, hb.pool, done)


@pytest.mark.parametrize("source", ["contiguous", "permuted"])
def test_slice_and_concatenate_keep_token_layer_plane_order(source, lib=None):
    spec = tagged_spec(source, "token")
    hb = host_buffers(spec, payload="tags")
    b = batch_of(hb, lib)
    hit0 = _cumsum0(spec.t_hit)
    tok0 = _cumsum0(spec.t_all())
    for layer in range(spec.L):
        st, hit_layer = b.slice_layer(layer)
        assert st == oracle.OK
        tags, uniform = decode_rows(hit_layer, spec.Rp)
        assert np.all(uniform)
        tags = tags.reshape(-1, spec.P, 4)
        assert tags.shape[0] == sum(spec.t_hit)
        for r, th in enumerate(spec.t_hit):
            for t in range(th):
                for p in range(spec.P):
                    assert np.array_equal(tags[hit0[r] + t, p], tag(r, t, layer, p, 0))
        st, complete = b.concatenate_tokens(layer, hit_layer)
        assert st == oracle.OK
        ctags, uniform = decode_rows(complete, spec.Rp)
        assert np.all(uniform)
        ctags = ctags.reshape(-1, spec.P, 4)
        for r, (th, tm) in enumerate(zip(spec.t_hit, spec.t_miss)):
            for t in range(th + tm):
                for p in range(spec.P):
                    assert np.array_equal(ctags[tok0[r] + t, p], tag(r, t, layer, p, int(t >= th)))
        # merge_scatter's complete_layer output is the same
        st, comp2 = b.merge_scatter(layer, hb.pool, want_complete=True)
        assert st == oracle.OK and np.array_equal(comp2, complete)


def test_gather_objects_hold_blocks_in_table_order(lib=None):
    spec = tagged_spec("permuted", "layer")
    hb = host_buffers(spec, payload="tags")
    b = batch_of(hb, lib)
    sent_row = np.frombuffer(bytes([SENT]) * 16, np.int32)
    for layer in range(spec.L):
        assert b.merge_scatter(layer, hb.pool)[0] == oracle.OK
        assert b.gather_objects(layer, hb.pool) == oracle.OK
    for r, q in enumerate(hb.layout.requests):
        th, ta = q.t_hit, q.t_hit + q.t_miss
        nblk = -(-ta // spec.B)
        region = hb.objects[q.obj_off:q.obj_off + spec.L * q.obj_layer_stride]
        tags, uniform = decode_rows(region, spec.Rp)
        assert np.all(uniform)
        tags = tags.reshape(spec.L, spec.P, nblk, spec.B, 4)
        for l in range(spec.L):
            for p in range(spec.P):
                for j in range(nblk):
                    for s in range(spec.B):
                        t = j * spec.B + s
                        want = tag(r, t, l, p, int(t >= th)) if t < ta else sent_row
                        assert np.array_equal(tags[l, p, j, s], want)
    assert np.all(hb.objects[hb.layout.obj_bytes:] == SENT)


def test_block_major_objects_form_one_file_of_2L_objects_per_block(lib=None):
    """Tutti 设计一 §3.1: one GPU file per KV block, holding 2L objects (a K and a V
    object per layer); 伪代码 1 addresses object (file, layer) at file x file stride +
    layer x per-layer size.  Decode every file back to (request, token, layer, plane)."""
    spec = workloads.custom_spec(L=3, P=2, B=4, Rp=32, **RAGGED, table="perm",
                                 source="permuted", seed=11, objects="block")
    hb = host_buffers(spec, payload="tags")
    b = batch_of(hb, lib)
    for layer in range(spec.L):
        assert b.merge_scatter(layer, hb.pool)[0] == oracle.OK
        assert b.gather_objects(layer, hb.pool) == oracle.OK
    sent_row = np.frombuffer(bytes([SENT]) * 16, np.int32)
    obj_bytes = spec.B * spec.Rp
    files = 0
    for r, q in enumerate(hb.layout.requests):
        th, ta = q.t_hit, q.t_hit + q.t_miss
        nblk = -(-ta // spec.B)
        for j in range(nblk):
            f0 = q.obj_off + j * q.obj_block_stride
            file_bytes = hb.objects[f0:f0 + 2 * spec.L * obj_bytes]
            assert file_bytes.size == 2 * spec.L * obj_bytes  # 2L objects per file
            tags, uniform = decode_rows(file_bytes, spec.Rp)
            assert np.all(uniform)
            tags = tags.reshape(spec.L, spec.P, spec.B, 4)
            for l in range(spec.L):
                for p in range(spec.P):
                    for s_ in range(spec.B):
                        t = j * spec.B + s_
                        want = tag(r, t, l, p, int(t >= th)) if t < ta else sent_row
                        assert np.array_equal(tags[l, p, s_], want)
            files += 1
    assert files == int(spec.nblk().sum())
    assert np.all(hb.objects[hb.layout.obj_bytes:] == SENT)
    # scatter-back from the files restores the pool
    before = hb.pool.copy()
    hb.pool[:] = SENT
    for layer in range(spec.L):
        assert b.scatter_back(layer, hb.pool) == oracle.OK
    assert np.array_equal(hb.pool, before)


# --------------------------------------------------------------------------
# Special cases that reduce to numpy slicing
# --------------------------------------------------------------------------

def test_identity_table_pool_is_a_reshape_of_complete_layer(lib=None):
    L, P, B, Rp, th, tm = 4, 2, 8, 48, 40, 24
    spec = workloads.custom_spec(L=L, P=P, B=B, Rp=Rp, t_hit=[th], t_miss=[tm],
                                 n_pool=(th + tm) // B, table="identity")
    hb = host_buffers(spec)
    b = batch_of(hb, lib)
    full = hb.hit[:th * L * P * Rp].reshape(th, L, P, Rp)
    miss = hb.miss[:L * tm * P * Rp].reshape(L, tm, P, Rp)
    for layer in range(L):
        assert b.merge_scatter(layer, hb.pool)[0] == oracle.OK
        assert b.gather_objects(layer, hb.pool) == oracle.OK
    pool = hb.pool[:hb.layout.pool_bytes].reshape(L, P, spec.n_pool * B, Rp)
    objs = hb.objects[:hb.layout.obj_bytes].reshape(L, P, spec.n_pool * B, Rp)
    for layer in range(L):
        for p in range(P):
            want = np.concatenate([full[:, layer, p], miss[layer, :, p]])
            assert np.array_equal(pool[layer, p], want)
            assert np.array_equal(objs[layer, p], want)
    hl = b.slice_layer(1)[1].reshape(th, P, Rp)
    assert np.array_equal(hl, full[:, 1])


def test_scatter_back_after_gather_restores_the_pool(lib=None):
    spec = tagged_spec("permuted", "layer")
    hb = host_buffers(spec)
    b = batch_of(hb, lib)
    for layer in range(spec.L):
        b.merge_scatter(layer, hb.pool)
        b.gather_objects(layer, hb.pool)
    before = hb.pool.copy()
    hb.pool[:] = SENT
    for layer in range(spec.L):
        assert b.scatter_back(layer, hb.pool) == oracle.OK
    assert np.array_equal(hb.pool, before)
    # and gather after scatter-back reproduces the objects
    objs = hb.objects.copy()
    hb.objects[:hb.layout.obj_bytes] = 0
    for layer in range(spec.L):
        b.gather_objects(layer, hb.pool)
    assert np.array_equal(hb.objects, objs)


# --------------------------------------------------------------------------
# Brute force on tiny inputs (pure Python, independent of the C loops)
# --------------------------------------------------------------------------

def brute(spec, hb, layer, pool, objects):
    """Byte-level restatement: returns (hit_layer, complete_layer) and updates pool,
    then gathers objects from the updated pool."""
    lay, R, Rp, B = hb.layout, spec.R, spec.Rp, spec.B
    hit_rows, comp_rows = [], []
    tab0 = 0
    for r, q in enumerate(lay.requests):
        ta = q.t_hit + q.t_miss
        nblk = -(-ta // B)
        tbl = hb.tables[tab0:tab0 + nblk]
        for t in range(ta):
            if t < q.t_hit:
                j, s = t // B, t % B
                blk = j if q.src_table_off < 0 else hb.src_tables[q.src_table_off + j]
                a = (q.hit_off + int(blk) * q.hit_block_stride + s * q.hit_token_stride
                     + layer * q.hit_layer_stride)
                row = hb.hit[a:a + R]
                hit_rows.append(row)
            else:
                a = q.miss_off + (t - q.t_hit) * q.miss_token_stride + layer * q.miss_layer_stride
                row = hb.miss[a:a + R]
            comp_rows.append(row)
            for p in range(spec.P):
                d = ((((layer * spec.P) + p) * spec.n_pool + int(tbl[t // B])) * B + t % B) * Rp
                pool[d:d + Rp] = row[p * Rp:(p + 1) * Rp]
        for p in range(spec.P):
            for j in range(nblk):
                src = (((layer * spec.P + p) * spec.n_pool + int(tbl[j])) * B) * Rp
                dst = q.obj_off + layer * q.obj_layer_stride + (p * nblk + j) * B * Rp
                objects[dst:dst + B * Rp] = pool[src:src + B * Rp]
        tab0 += nblk
    cat = lambda rows: np.concatenate(rows) if rows else np.zeros(0, np.uint8)
    return cat(hit_rows), cat(comp_rows)


@pytest.mark.parametrize("case", range(6))
def test_oracle_matches_brute_force(case, lib=None):
    g = np.random.default_rng(100 + case)
    n = int(g.integers(1, 5))
    P = int(g.integers(1, 3))
    B = int(g.choice([1, 2, 4, 16]))
    spec = workloads.custom_spec(
        L=int(g.integers(1, 4)), P=P, B=B, Rp=int(g.choice([16, 32, 48])),
        t_hit=g.integers(0, 40, n), t_miss=g.integers(0, 20, n),
        table=str(g.choice(["perm", "fragmented"])), source=str(g.choice(["contiguous", "permuted"])),
        miss_order=str(g.choice(["layer", "token"])), seed=200 + case)
    hb = host_buffers(spec, seed=300 + case)
    b = batch_of(hb, lib)
    pool_bf = hb.pool.copy()
    obj_bf = hb.objects.copy()
    for layer in range(spec.L):
        st, hit_layer = b.slice_layer(layer)
        assert st == oracle.OK
        st, comp = b.merge_scatter(layer, hb.pool, want_complete=True)
        assert st == oracle.OK
        assert b.gather_objects(layer, hb.pool) == oracle.OK
        want_hit, want_comp = brute(spec, hb, layer, pool_bf, obj_bf)
        assert np.array_equal(hit_layer, want_hit)
        assert np.array_equal(comp, want_comp)
        assert np.array_equal(hb.pool, pool_bf)
        assert np.array_equal(hb.objects, obj_bf)


# --------------------------------------------------------------------------
# Plan
# --------------------------------------------------------------------------

def test_plan_prefix_sums_and_work_list(lib=None):
    spec = tagged_spec()
    hb = host_buffers(spec)
    plan = batch_of(hb, lib).plan()
    assert plan["status"] == oracle.OK
    ta = spec.t_all()
    nblk = np.array([-(-int(x) // spec.B) for x in ta])
    assert np.array_equal(plan["tok_off"], _cumsum0(ta))
    assert np.array_equal(plan["hit_off"], _cumsum0(spec.t_hit))
    assert np.array_equal(plan["blk_off"], _cumsum0(nblk))
    pairs = [(r, j) for r in range(spec.n_req) for j in range(int(nblk[r]))]
    assert plan["n_items"] == len(pairs)
    assert list(zip(plan["item_req"].tolist(), plan["item_blk"].tolist())) == pairs


def test_plan_flags_planted_errors(lib=None):
    spec = tagged_spec()
    hb = host_buffers(spec)
    n = len(hb.tables)
    # out of range pool block id at flat index 5 and 9 -> ERANGE, detail 5
    t = hb.tables.copy(); t[9] = spec.n_pool; t[5] = -1
    hb2 = host_buffers(spec); hb2.tables = t
    p = batch_of(hb2, lib).plan()
    assert (p["status"], p["detail"]) == (oracle.ERANGE, 5)
    # duplicate ids -> EDUP with the smallest duplicated id; without the check, OK
    t = hb.tables.copy(); t[7] = t[2]; t[n - 1] = t[0]
    hb2.tables = t
    p = batch_of(hb2, lib).plan()
    assert (p["status"], p["detail"]) == (oracle.EDUP, int(min(t[2], t[0])))
    assert batch_of(hb2, lib).plan(check_injective=False)["status"] == oracle.OK
    # both -> the larger code (EDUP)
    t[3] = spec.n_pool + 4
    hb2.tables = t
    assert batch_of(hb2, lib).plan()["status"] == oracle.EDUP
    # capacity
    p = batch_of(hb, lib).plan(capacity=n - 1)
    assert (p["status"], p["detail"]) == (oracle.ERANGE, n)
    # a full-block id outside the source buffer -> ERANGE at that work item
    st = hb.src_tables.copy()
    st[2] = 1000
    hb3 = host_buffers(spec); hb3.src_tables = st
    p = batch_of(hb3, lib).plan()
    # source table entry 2 belongs to request 0 (the first with hits), block 2 -> item 2
    assert (p["status"], p["detail"]) == (oracle.ERANGE, 2)


def test_plan_rejects_negative_counts(lib=None):
    spec = tagged_spec()
    hb = host_buffers(spec)
    reqs = list(hb.layout.requests)
    import dataclasses
    reqs[2] = dataclasses.replace(reqs[2], t_miss=-1)
    b = oracle.Batch(geom_of(spec), reqs, hb.hit, hb.miss, hb.objects, hb.tables,
                     hb.src_tables, lib=lib)
    p = b.plan()
    assert (p["status"], p["detail"]) == (oracle.EINVAL, 2)


# --------------------------------------------------------------------------
# Edge cases
# --------------------------------------------------------------------------

def test_empty_batch_and_degenerate_requests(lib=None):
    spec = workloads.custom_spec(L=2, P=2, B=4, Rp=16, t_hit=[], t_miss=[])
    hb = host_buffers(spec)
    b = batch_of(hb, lib)
    p = b.plan()
    assert p["status"] == oracle.OK and p["n_items"] == 0
    assert b.merge_scatter(0, hb.pool)[0] == oracle.OK
    assert np.all(hb.pool == SENT)
    # only-miss, only-hit, empty, shorter-than-a-block
    spec = workloads.custom_spec(L=2, P=2, B=8, Rp=16, t_hit=[0, 12, 0, 3], t_miss=[9, 0, 0, 2],
                                 seed=5)
    hb = host_buffers(spec, payload="tags")
    b = batch_of(hb, lib)
    assert b.plan()["n_items"] == 2 + 2 + 0 + 1
    for layer in range(2):
        assert b.merge_scatter(layer, hb.pool)[0] == oracle.OK
    check_pool(spec, hb.pool, {0, 1})
