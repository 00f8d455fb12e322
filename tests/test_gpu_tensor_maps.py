"""The plan's tensor maps, checked without running a single tensor load.

kvl_batch_plan builds, on the device, tensor maps for each strided row source of a
request (hit rows read a plane at a time, hit rows read a whole token row at a time
for the slice, miss rows; each with a box of a whole segment's rows and one of a
block's tail), by editing a host-encoded template with
`tensormap.replace`.  Here every map the plan wrote is compared, byte for byte, with
the map the driver's own host encoder (cuTensorMapEncodeTiled) makes for the view
that the request's strides declare, and every item record's map flags and
coordinates with their definition.  The view rules are restated below from the
library's documentation of the maps: 8-byte elements; dim 0 one chunk of a token
row, dim 1 the chunks of the row, dims 2 and 3 tokens and layers (smaller stride
first), dim 4 full blocks of a table source; the box one plane row (or one token
row for the slice) wide and one segment of rows high; a map only where each stride
is at least the extent below it and some dim spans at least 1 MiB.

Most cases are plan-only batches whose source addresses are placeholders: the plan
kernels check a source pointer's alignment but never read through it, so views of
any span (up to tens of GB) are checked without allocating them.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests._device import device_batch
from tests._host import host_buffers

pytestmark = pytest.mark.gpu

STAGE = 32 * 1024
MAX_STRIDE = 1 << 40
MIN_SPAN = 1 << 20
MAP_HIT, MAP_SLICE, MAP_MISS, MAP_HIT_TAIL, MAP_SLICE_TAIL, MAP_MISS_TAIL = range(6)
KINDS = 6          # maps per request
TAIL = 3           # a kind's block-tail kind is kind + TAIL
F_HIT_LAYER_FIRST, F_MISS_LAYER_FIRST = 64, 128   # record flags beside bit `kind`


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    kvl.lib()


def chunk_bytes(Rp):
    for c in range((min(Rp, 2048) // 16) * 16, 15, -16):
        if Rp % c == 0:
            return c
    return 0


def seg_rows(B, w):
    return min(B, STAGE // w)


def kind_width(kind, P, Rp):
    return P * Rp if kind in (MAP_SLICE, MAP_SLICE_TAIL) else Rp


def kind_rows(kind, B, P, Rp):
    """Box rows: a whole segment, or a block's tail (B mod the segment rows)."""
    m = seg_rows(B, kind_width(kind, P, Rp))
    return m if kind < TAIL else (B % m if m else 0)


def map_ops(P, B, Rp):
    C, R = chunk_bytes(Rp), P * Rp
    ops = 0
    for k in range(KINDS):
        w = kind_width(k, P, Rp)
        if C and w <= STAGE and w // C <= 256 and 1 <= kind_rows(k, B, P, Rp) <= 256:
            ops |= 1 << k
    return ops


def view(base, n_tok, ts, L, ls, n_blk, bs, R, C, W, rows):
    """(dims, strides, box, layer_first) of a map over these rows, or None."""
    if base == 0 or n_tok < rows or L < 1 or n_blk < 1 or n_tok >= 2**31 or n_blk >= 2**31:
        return None
    layer_first = L > 1 and (n_tok == 1 or ls < ts)
    e_in, e_out = (L, n_tok) if layer_first else (n_tok, L)
    s_in, s_out = (ls, ts) if layer_first else (ts, ls)
    if e_in == 1:
        s_in = R
    if s_in < R or s_in >= MAX_STRIDE:
        return None
    if e_out == 1:
        s_out = e_in * s_in
    elif s_out < e_in * s_in:
        return None
    if s_out >= MAX_STRIDE:
        return None
    if n_blk == 1:
        bs = e_out * s_out
    elif bs < e_out * s_out:
        return None
    if bs >= MAX_STRIDE:
        return None
    dims = [C // 8, R // C, e_in, e_out, n_blk]
    if max((d - 1) * st for d, st in zip(dims, [8, C, s_in, s_out, bs])) < MIN_SPAN:
        return None
    strides = [C, s_in, s_out, bs]
    box = [C // 8, W // C, 1 if layer_first else rows, rows if layer_first else 1, 1]
    return dims, strides, box, layer_first


def expected_maps(q, L, P, B, Rp):
    """{kind: view} and the record flags of request q (a kvl_request as a numpy record)."""
    ops, C, R = map_ops(P, B, Rp), chunk_bytes(Rp), P * Rp
    out, flags = {}, 0
    t_hit, t_miss = int(q["t_hit"]), int(q["t_miss"])
    if ops and t_hit > 0:
        ts, bs = int(q["hit_token_stride"]), int(q["hit_block_stride"])
        n_tok = n_blk = 0
        if int(q["hit_src_table"]):
            n_tok, n_blk = B, int(q["hit_src_blocks"])
        elif t_hit <= B or (ts > 0 and bs == B * ts):
            n_tok, n_blk = t_hit, 1
        if n_tok:
            args = (int(q["hit_src"]), n_tok, ts, L, int(q["hit_layer_stride"]), n_blk, bs, R, C)
            for k in (MAP_HIT, MAP_SLICE, MAP_HIT_TAIL, MAP_SLICE_TAIL):
                v = view(*args, kind_width(k, P, Rp), kind_rows(k, B, P, Rp)) \
                    if ops & (1 << k) else None
                if v:
                    out[k] = v
                    flags |= (1 << k) | (F_HIT_LAYER_FIRST if v[3] else 0)
    if t_miss > 0:
        for k in (MAP_MISS, MAP_MISS_TAIL):
            v = view(int(q["miss_src"]), t_miss, int(q["miss_token_stride"]), L,
                     int(q["miss_layer_stride"]), 1, 0, R, C, Rp, kind_rows(k, B, P, Rp)) \
                if ops & (1 << k) else None
            if v:
                out[k] = v
                flags |= (1 << k) | (F_MISS_LAYER_FIRST if v[3] else 0)
    return out, flags


_encode = None


def host_encode(base, dims, strides, box):
    """128 bytes of cuTensorMapEncodeTiled for this view (the plan's template options)."""
    global _encode
    if _encode is None:
        torch.cuda.init()
        f = ctypes.CDLL("libcuda.so.1").cuTensorMapEncodeTiled
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_void_p,
                      ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                      ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _encode = f
    raw = ctypes.create_string_buffer(256)
    addr = (ctypes.addressof(raw) + 63) & ~63   # a tensor map is 64-byte aligned
    u64, u32 = ctypes.c_uint64, ctypes.c_uint32
    rc = _encode(addr, 4, 5, base, (u64 * 5)(*dims), (u64 * 4)(*strides), (u32 * 5)(*box),
                 (u32 * 5)(1, 1, 1, 1, 1), 0, 0, 2, 0)  # UINT64; no interleave or swizzle;
    assert rc == 0, f"cuTensorMapEncodeTiled failed ({rc})"  # L2 promotion 128 B; zero fill
    return np.frombuffer(ctypes.string_at(addr, 128), np.uint8)


def check_plan(g, n_req, reqs, d_reqs, tables, src_tables, d_plan, layout):
    """Compare every map and item record of a built plan with their definition.

    reqs: the kvl_request records (numpy); src_tables: {request: numpy table}.
    Returns the number of maps compared."""
    L, P, B, Rp = g.n_layers, g.n_planes, g.block_tokens, g.plane_row_bytes
    plan = d_plan.cpu().numpy()
    base = d_plan.data_ptr()
    maps_at = ((base + layout[10] + 127) & ~127) - base
    n_maps, flags_of = 0, []
    for r in range(n_req):
        q = reqs[r]
        want, flags = expected_maps(q, L, P, B, Rp)
        flags_of.append(flags)
        for kind, (dims, strides, box, _) in want.items():
            at = maps_at + (r * KINDS + kind) * 128
            got = plan[at:at + 128]
            miss = kind in (MAP_MISS, MAP_MISS_TAIL)
            exp = host_encode(int(q["miss_src"] if miss else q["hit_src"]), dims, strides, box)
            assert np.array_equal(got, exp), (r, kind, dims, strides, box,
                                              np.nonzero(got != exp)[0])
            n_maps += 1
    # item records: words 26..29 are the hit block / hit token / miss token
    # coordinates of slot 0 and the request's map flags
    t_hit = reqs["t_hit"].astype(np.int64)
    nblk = -(-(t_hit + reqs["t_miss"]) // B)
    n_items = int(nblk.sum())
    recs = plan[256:256 + 128 * n_items].view(np.int32).reshape(-1, 32)
    req = np.repeat(np.arange(n_req), nblk)
    j = np.arange(n_items) - np.repeat(np.cumsum(nblk) - nblk, nblk)
    assert np.array_equal(recs[:, 29], np.asarray(flags_of, np.int32)[req])
    assert np.array_equal(recs[:, 28], (j * B - t_hit[req]).astype(np.int32))
    for r in range(n_req):
        sel = (req == r) & (j * B < t_hit[req])
        jj = j[sel]
        if r in src_tables:
            assert np.array_equal(recs[sel, 26], src_tables[r][jj])
            assert not recs[sel, 27].any()
        else:
            assert not recs[sel, 26].any()
            assert np.array_equal(recs[sel, 27], (jj * B).astype(np.int32))
    return n_maps


def plan_of(g, reqs, tables, src_dev):
    """Build the plan of `reqs` (numpy kvl_request records) on the device."""
    import layer_wise_paged_gb300 as kvl
    n = len(reqs)
    d_reqs = torch.from_numpy(np.ascontiguousarray(reqs).view(np.uint8).copy()).cuda()
    d_tab = torch.from_numpy(np.ascontiguousarray(tables, np.int32)).cuda()
    nbytes = kvl.kvl_plan_bytes(g, n)
    d_plan = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    st = kvl.kvl_batch_plan(g, n, d_reqs.data_ptr(), d_tab.data_ptr(), 1, d_plan.data_ptr(),
                            nbytes)
    assert st == kvl.KVL_OK
    assert kvl.kvl_read_status(d_plan.data_ptr()) == (0, 0)
    return d_reqs, d_plan, kvl.kvl_plan_layout(g, n), (d_tab, src_dev)


PLACEHOLDER = 1 << 44  # an address range no buffer of this process has


def synthetic_case(seed):
    """A random geometry and batch whose sources sit at placeholder addresses."""
    import layer_wise_paged_gb300 as kvl
    from layer_wise_paged_gb300 import REQUEST_DTYPE
    g = np.random.default_rng(seed)
    L = int(g.choice([1, 2, 5, 32, 61]))
    P = int(g.integers(1, 3))
    Rp = int(g.choice([16, 48, 256, 1152, 2048, 4096, 16384]))
    B = int(g.choice([1, 3, 16, 64]))
    R = P * Rp
    n = int(g.choice([1, 3, 9]))
    reqs = np.zeros(n, REQUEST_DTYPE)
    src_tables, src_dev = {}, []
    addr = PLACEHOLDER
    for r in range(n):
        cap = 12_000 * B  # at most 12,000 blocks per request
        th = int(g.choice([0, 1, B, g.integers(1, 3000), g.integers(1, 200_000)]))
        tm = int(g.choice([0, 1, g.integers(1, 3000), g.integers(1, 60_000)]))
        th, tm = min(th, cap // 2), min(tm, cap // 2)
        nsrc = -(-th // B)
        q = reqs[r]
        q["t_hit"], q["t_miss"] = th, tm
        pad = 16 * int(g.integers(0, 4))
        kind = str(g.choice(["contiguous", "permuted", "layer_major", "gapped", "overlap"]))
        if kind == "contiguous":
            ts, ls = L * R + pad, R
            bs, blocks = B * ts, nsrc
        elif kind == "permuted":
            ts, ls = L * R, R
            bs, blocks = B * L * R + pad, nsrc + int(g.integers(0, 5))
        elif kind == "layer_major":
            ts, ls = R, max(th, 1) * R + pad
            bs, blocks = B * ts, nsrc
        elif kind == "gapped":     # blocks not B rows apart, and no table: no map
            ts, ls = L * R, R
            bs, blocks = B * ts + 16, nsrc
        else:                      # every layer on the same rows: no map when L > 1
            ts, ls = R, 0
            bs, blocks = B * ts, nsrc
        q["hit_token_stride"], q["hit_layer_stride"], q["hit_block_stride"] = ts, ls, bs
        q["hit_src_blocks"] = blocks
        if th:
            q["hit_src"] = addr
            addr += max(blocks, 1) * max(bs, B * ts, 16) + L * R * 2 + 16 * int(g.integers(0, 8))
            if kind == "permuted":
                tab = g.permutation(blocks)[:nsrc].astype(np.int32)
                t = torch.from_numpy(tab).cuda()
                src_dev.append(t)
                src_tables[r] = tab
                q["hit_src_table"] = t.data_ptr()
        mk = str(g.choice(["layer", "token", "overlap", "huge"]))
        mts, mls = {"layer": (R, tm * R), "token": (L * R, R), "overlap": (R, 0),
                    "huge": (R, 1 << 40)}[mk]
        q["miss_token_stride"], q["miss_layer_stride"] = mts, mls
        if tm:
            q["miss_src"] = addr
            addr += tm * mts * 2 + L * R * 2 + 16 * int(g.integers(0, 8))
    nblk = -(-(reqs["t_hit"].astype(np.int64) + reqs["t_miss"]) // B)
    N = max(1, int(nblk.sum()))
    tables = g.permutation(N).astype(np.int32)[:max(1, int(nblk.sum()))]
    geo = kvl.geom(L, P, B, Rp, N)
    return geo, reqs, tables, src_tables, src_dev


CASES = 40


@pytest.mark.parametrize("case", range(CASES))
def test_plan_maps_equal_the_host_encoder(case):
    geo, reqs, tables, src_tables, src_dev = synthetic_case(4100 + case)
    d_reqs, d_plan, layout, keep = plan_of(geo, reqs, tables, src_dev)
    check_plan(geo, len(reqs), reqs, d_reqs, tables, src_tables, d_plan, layout)


def test_synthetic_cases_cover_every_map_kind_and_order():
    """The random cases above build maps of each kind, the whole-segment kinds in
    both dim orders."""
    seen = set()
    for case in range(CASES):
        geo, reqs, _, _, _ = synthetic_case(4100 + case)
        for q in reqs:
            want, _ = expected_maps(q, geo.n_layers, geo.n_planes, geo.block_tokens,
                                    geo.plane_row_bytes)
            seen |= {(k, v[3]) for k, v in want.items()}
    assert {k for k, _ in seen} == set(range(KINDS))
    assert {(k, o) for k in (MAP_HIT, MAP_SLICE, MAP_MISS) for o in (False, True)} <= seen


def test_workload_shapes_get_maps():
    """Requests shaped like the benchmark's workloads, over real buffers, each get
    all their maps."""
    for name, kw in {
        "llama3_8b_agentic": dict(L=32, P=2, B=16, Rp=2048, t_hit=[3000], t_miss=[77]),
        "qwen3_32b_long": dict(L=8, P=2, B=64, Rp=2048, t_hit=[1280], t_miss=[300],
                               source="permuted"),
        "latent_batch": dict(L=61, P=1, B=64, Rp=1152, t_hit=[1700, 900], t_miss=[130, 2000]),
        "many_small": dict(L=32, P=2, B=16, Rp=2048, t_hit=[300, 270], t_miss=[16, 250]),
    }.items():
        spec = workloads.custom_spec(name, **kw, table="perm", seed=77)
        hb = host_buffers(spec)
        gb, _ = device_batch(spec, hb)
        gb.plan()
        assert gb.status() == (0, 0)
        from layer_wise_paged_gb300 import REQUEST_DTYPE
        reqs = gb.d_reqs.cpu().numpy()[:gb.n_req * 112].view(REQUEST_DTYPE)
        src = {}
        for r, lq in enumerate(hb.layout.requests):
            if lq.src_table_off >= 0:
                nsrc = -(-lq.t_hit // spec.B)
                src[r] = hb.src_tables[lq.src_table_off:lq.src_table_off + nsrc]
        n = check_plan(gb.g, gb.n_req, reqs, gb.d_reqs, hb.tables, src, gb.d_plan, gb.layout)
        # three kinds per request, and the three block-tail kinds where blocks have a
        # tail (the latent batch's 64-token blocks of 1,152-byte rows: 28 + 28 + 8)
        tails = sum(kind_rows(k, spec.B, spec.P, spec.Rp) > 0 for k in range(TAIL, KINDS))
        assert n == (3 + tails) * spec.n_req, name


def test_small_or_overlapping_sources_get_no_map():
    """Sources a map cannot express exactly, or that span under 1 MiB, keep the
    per-row loads: a miss layer stride of 0 with several layers (every layer reads
    the same rows), a hit source without a table whose blocks are not B rows apart,
    and the tiny workload."""
    spec = workloads.custom_spec(L=3, P=2, B=16, Rp=2048, t_hit=[400], t_miss=[300],
                                 table="perm", seed=5)
    hb = host_buffers(spec)
    lq = hb.layout.requests[0]
    lq.miss_layer_stride = 0
    lq.hit_block_stride = lq.hit_block_stride + 512
    hb.hit = np.concatenate([hb.hit, np.zeros(16384, np.uint8)])
    gb, _ = device_batch(spec, hb)
    gb.plan()
    assert gb.status() == (0, 0)
    assert gb.d_plan.cpu().numpy()[256:256 + 128].view(np.int32)[29] == 0
    tiny = workloads.get_spec("tiny")
    hb = host_buffers(tiny)
    gb, _ = device_batch(tiny, hb)
    gb.plan()
    assert gb.status() == (0, 0)
    recs = gb.d_plan.cpu().numpy()[256:256 + 128 * gb.n_items].view(np.int32).reshape(-1, 32)
    assert not recs[:, 29].any()
