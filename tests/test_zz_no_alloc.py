"""kvl_batch_plan_static_scratch: the plan builder for callers that cannot allocate.

Some callers cannot call cudaMalloc (for example an engine whose allocator already
owns the HBM); this entry point takes its only scratch, the injectivity bitmap, from
a fixed array inside the library.  The test calls it through the C ABI twice in a
row and checks that each time its plan and status equal those of kvl_batch_plan,
byte for byte (the plan holds only integers), on a clean batch and on a batch with a
duplicate block id (which exercises the shared bitmap), and that the copy kernels
accept its plan.  This file is collected last on purpose; it also passes alone.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import layer_wise_paged_gb300 as kvl
import workloads
from tests._device import device_batch
from tests._host import host_buffers

pytestmark = pytest.mark.gpu

SPEC = workloads.custom_spec(L=2, P=2, B=16, Rp=256, t_hit=[300, 0, 77, 41, 900],
                             t_miss=[20, 33, 0, 5, 64], table="perm", source="permuted",
                             seed=4242)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvl.build()
    kvl.lib()


def _plan_bytes_used(plan_u8, off, n_req, n_items):
    """The bytes of a plan that carry results: header fields, offsets, work list,
    item records and claim counters."""
    p = plan_u8.cpu().numpy()
    hdr = p[:144]
    return dict(
        status=hdr[:4].copy(), counts=hdr[8:40].copy(), detail=hdr[64:128].copy(),
        tok_off=p[off[1]:off[1] + 8 * (n_req + 1)].copy(),
        hit_off=p[off[2]:off[2] + 8 * (n_req + 1)].copy(),
        blk_off=p[off[3]:off[3] + 8 * (n_req + 1)].copy(),
        item_req=p[off[4]:off[4] + 4 * n_items].copy(),
        item_blk=p[off[5]:off[5] + 4 * n_items].copy(),
        records=p[off[6]:off[6] + 128 * n_items].copy(),
        counters=p[off[7]:off[7] + 8 * 4 * SPEC.L].copy())


def _compare_twice(tables_override=None):
    hb = host_buffers(SPEC)
    if tables_override is not None:
        hb.tables = tables_override(hb.tables.copy())
    gb, d = device_batch(SPEC, hb)
    stream = torch.cuda.current_stream().cuda_stream
    gb.plan()
    want_status = gb.status()
    off = gb.layout
    n_items = min(gb.n_items, SPEC.n_pool)
    want = _plan_bytes_used(gb.d_plan, off, gb.n_req, n_items)

    small = torch.empty(off[8], dtype=torch.uint8, device="cuda")
    for call in range(2):
        small.fill_(0x5A + call)  # stale bytes must not leak into the result
        st = kvl.kvl_batch_plan_static_scratch(gb.g, gb.n_req, gb.d_reqs.data_ptr(),
                                               gb.tables.data_ptr(), 1, small.data_ptr(),
                                               small.numel(), stream)
        assert st == kvl.KVL_OK
        assert kvl.kvl_read_status(small.data_ptr(), stream) == want_status, f"call {call}"
        got = _plan_bytes_used(small, off, gb.n_req, n_items)
        for k in want:
            assert np.array_equal(got[k], want[k]), f"call {call}: {k}"
    return gb, d, small, want_status


def test_static_scratch_plan_equals_kvl_batch_plan_on_two_calls():
    gb, d, small, status = _compare_twice()
    assert status == (0, 0)
    # the copy kernels accept it: merge-scatter with either plan gives the same pool
    stream = torch.cuda.current_stream().cuda_stream
    pool_ref = d.pool.clone()
    for layer in range(SPEC.L):
        gb.merge_scatter(layer, pool_ref)
        assert kvl.kvl_merge_scatter_paged(gb.g, small.data_ptr(), small.numel(),
                                           gb.d_reqs.data_ptr(), gb.tables.data_ptr(), layer, 1,
                                           d.pool.data_ptr(), None, None, stream) == kvl.KVL_OK
    torch.cuda.synchronize()
    assert torch.equal(d.pool, pool_ref)
    assert kvl.kvl_read_status(small.data_ptr(), stream) == (0, 0)


def test_static_scratch_plan_finds_the_same_duplicate_on_two_calls():
    def dup(t):
        t[9] = t[3]
        return t
    _, _, _, status = _compare_twice(dup)
    assert status[0] == kvl.KVL_EDUP


def test_static_scratch_plan_rejects_pools_beyond_its_array():
    """The refusal comes from the array's limit, not from another check: the geometry
    itself is valid (kvl_plan_bytes accepts it), a pool of exactly the limit passes the
    limit check and is stopped by the next one (a misaligned plan: KVL_EALIGN), and one
    block more is refused before that check is reached (KVL_EINVAL)."""
    limit = kvl.KVL_STATIC_SCRATCH_POOL_BLOCKS
    big = kvl.geom(SPEC.L, SPEC.P, SPEC.B, SPEC.Rp, limit + 1)
    at = kvl.geom(SPEC.L, SPEC.P, SPEC.B, SPEC.Rp, limit)
    assert kvl.kvl_plan_bytes(big, 1) != 0 and kvl.kvl_plan_bytes(at, 1) != 0
    fake = 1 << 20  # never dereferenced: every call below is refused on the host
    huge = 1 << 40
    call = kvl.kvl_batch_plan_static_scratch
    assert call(big, 1, fake, fake, 1, fake, huge) == kvl.KVL_EINVAL
    assert call(big, 1, fake, fake, 1, fake + 8, huge) == kvl.KVL_EINVAL  # limit first
    assert call(at, 1, fake, fake, 1, fake + 8, huge) == kvl.KVL_EALIGN   # past the limit
    # at the limit, a plan one byte short of the bitmap-free plan is refused too
    need = kvl.kvl_plan_layout(at, 1)[8]
    assert call(at, 1, fake, fake, 1, fake, need - 1) == kvl.KVL_EINVAL
