"""Error paths on the GPU: every failure is a status code, never a fault.

Host-visible problems return at once and launch nothing; device-visible ones are
recorded in the plan's status word (compared with the oracle's verdict for the same
planted error), the offending work is skipped, and later calls on a failed plan
leave every buffer untouched.  Every planted error here keeps all accesses in bounds.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import layer_wise_paged_gb300 as kvl
import oracle
import workloads
from tests._device import device_batch
from tests._host import geom_of, host_buffers

pytestmark = pytest.mark.gpu

SPEC = workloads.custom_spec(L=2, P=2, B=4, Rp=32, t_hit=[10, 0, 7, 8], t_miss=[3, 5, 0, 1],
                             table="perm", source="permuted", seed=11)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kvl.build()
    kvl.lib()


def _both(hb, requests=None, check_injective=True):
    reqs = requests if requests is not None else hb.layout.requests
    hb.layout.requests = reqs
    gb, d = device_batch(SPEC, hb)
    gb.plan(check_injective=check_injective)
    ob = oracle.Batch(geom_of(SPEC), reqs, hb.hit, hb.miss, hb.objects, hb.tables, hb.src_tables)
    op = ob.plan(check_injective=check_injective)
    return gb, d, op


@pytest.mark.parametrize("kind", ["pool_range", "dup", "dup_and_range", "src_range", "neg"])
def test_plan_status_matches_oracle(kind):
    hb = host_buffers(SPEC)
    reqs = list(hb.layout.requests)
    if kind == "pool_range":
        hb.tables = hb.tables.copy(); hb.tables[9] = SPEC.n_pool; hb.tables[5] = -3
    elif kind == "dup":
        hb.tables = hb.tables.copy(); hb.tables[7] = hb.tables[2]
    elif kind == "dup_and_range":
        hb.tables = hb.tables.copy(); hb.tables[7] = hb.tables[2]; hb.tables[1] = 1 << 30
    elif kind == "src_range":
        hb.src_tables = hb.src_tables.copy(); hb.src_tables[4] = 99
    elif kind == "neg":
        reqs[3] = dataclasses.replace(reqs[3], t_hit=-2)
    gb, d, op = _both(hb, reqs)
    code, detail = gb.status()
    assert code != 0
    assert (code, detail) == (op["status"], op["detail"])
    # a failed plan makes every later call a no-op
    pool0 = d.pool.clone()
    objs0 = d.objects.clone()
    for layer in range(SPEC.L):
        gb.merge_scatter(layer, d.pool)
        gb.gather(layer, d.pool)
    assert torch.equal(d.pool, pool0) and torch.equal(d.objects, objs0)
    assert gb.status() == (code, detail)


def test_duplicates_pass_without_the_check():
    hb = host_buffers(SPEC)
    hb.tables = hb.tables.copy(); hb.tables[7] = hb.tables[2]
    gb, d, op = _both(hb, check_injective=False)
    assert gb.status() == (0, 0) and op["status"] == 0


def test_misaligned_request_fields_are_ealign():
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    host = kvl.pack_requests(hb.layout.requests, hit_base=d.hit.data_ptr(),
                             miss_base=d.miss.data_ptr(), obj_base=d.objects.data_ptr(),
                             src_table_base=d.src_tables.data_ptr())
    for field, delta, want in [("hit_src", 8, kvl.KVL_EALIGN), ("miss_token_stride", 4, kvl.KVL_EALIGN),
                               ("objects", 4, kvl.KVL_EALIGN)]:
        bad = host.copy()
        r = 0 if field != "miss_token_stride" else 1
        bad[r][field] = int(bad[r][field]) + delta
        gb.d_reqs.copy_(torch.from_numpy(bad.view(np.uint8).reshape(-1).copy()))
        gb.plan()
        assert gb.status() == (want, r), field
        pool0 = d.pool.clone()
        gb.merge_scatter(0, d.pool)
        assert torch.equal(d.pool, pool0)


def test_null_sources_are_einval():
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    host = kvl.pack_requests(hb.layout.requests, hit_base=0, miss_base=d.miss.data_ptr(),
                             obj_base=d.objects.data_ptr(), src_table_base=d.src_tables.data_ptr())
    gb.d_reqs.copy_(torch.from_numpy(host.view(np.uint8).reshape(-1).copy()))
    gb.plan()
    assert gb.status() == (kvl.KVL_EINVAL, 0)


def test_tables_edited_after_planning_take_effect_only_through_a_new_plan():
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    gb.plan()
    pool0 = d.pool.clone()
    gb.merge_scatter(0, pool0)
    # the plan resolved block ids when it was built: an edit alone changes nothing
    d.tables[6] = SPEC.n_pool + 1
    pool1 = d.pool.clone()
    gb.merge_scatter(0, pool1)
    assert gb.status() == (0, 0) and torch.equal(pool0, pool1)
    # a new plan sees the edit and refuses it
    gb.plan()
    assert gb.status() == (kvl.KVL_ERANGE, 6)


def test_missing_objects_pointer_is_einval_at_gather():
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    host = kvl.pack_requests(hb.layout.requests, hit_base=d.hit.data_ptr(),
                             miss_base=d.miss.data_ptr(), obj_base=0,
                             src_table_base=d.src_tables.data_ptr())
    gb.d_reqs.copy_(torch.from_numpy(host.view(np.uint8).reshape(-1).copy()))
    gb.plan()
    gb.merge_scatter(0, d.pool)
    assert gb.status() == (0, 0)
    gb.gather(0, d.pool)
    assert gb.status() == (kvl.KVL_EINVAL, 0)


def test_a_plan_that_fails_while_a_plan_ready_launch_waits_writes_nothing():
    """A launch with KVL_LAUNCH_PLAN_READY checks the plan before its dependency wait and
    reads the status word again after it.  Here the gather before it records
    KVL_EINVAL late in its run (the request without objects is the last one claimed),
    so the merge-scatter after it may find the plan sound before the wait and failed
    after it: either way it must write nothing to its (sentinel) pool."""
    spec = workloads.custom_spec(L=2, P=2, B=16, Rp=2048, t_hit=[12000, 9000, 20],
                                 t_miss=[300, 100, 4], table="perm", seed=31)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    host = kvl.pack_requests(hb.layout.requests, hit_base=d.hit.data_ptr(),
                             miss_base=d.miss.data_ptr(), obj_base=d.objects.data_ptr())
    host[2]["objects"] = 0  # the last request has no objects: its gather item fails
    gb.d_reqs.copy_(torch.from_numpy(host.view(np.uint8).reshape(-1).copy()))
    pool2 = torch.full_like(d.pool, workloads.SENTINEL)
    for rep in range(3):
        gb.plan()
        gb.merge_scatter(0, d.pool)
        assert gb.status() == (0, 0)
        gb.gather(0, d.pool)
        gb.merge_scatter(1, pool2, flags=kvl.KVL_LAUNCH_PLAN_READY)
        gb.gather(1, d.pool, flags=kvl.KVL_LAUNCH_PLAN_READY)
        assert gb.status() == (kvl.KVL_EINVAL, 2), rep
        assert bool((pool2 == workloads.SENTINEL).all()), f"repetition {rep}: a failed plan wrote"


def test_host_side_checks_return_without_launching():
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    gb.plan()
    g, plan, reqs, tabs = gb.g, gb.d_plan.data_ptr(), gb.d_reqs.data_ptr(), gb.tables.data_ptr()
    pool = d.pool.data_ptr()
    pb = gb.plan_bytes
    s = torch.cuda.current_stream().cuda_stream
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, SPEC.L, 1, pool, None, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, -1, 1, pool, None, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, SPEC.L + 1, pool, None, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool + 8, None, None, s) == kvl.KVL_EALIGN
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, 0, None, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_gather_layer_objects(g, plan, pb, reqs, tabs, 0, 1, pool, 2, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_slice_layer(g, plan, pb, reqs, 0, 1, 0, None, s) == kvl.KVL_EINVAL
    assert kvl.kvl_batch_plan(g, gb.n_req, reqs, tabs, 1, plan, gb.plan_bytes - 1, s) == kvl.KVL_EINVAL
    # a plan buffer smaller than the geometry's smallest plan: refused on the host, for
    # every op, with nothing launched (pool and status untouched)
    least = kvl.kvl_plan_layout(g, 0)[8]
    before = d.pool.clone()
    for small in (16, least - 16):
        assert kvl.kvl_slice_layer(g, plan, small, reqs, 0, 1, pool, None, s) == kvl.KVL_EINVAL
        assert kvl.kvl_merge_scatter_paged(g, plan, small, reqs, tabs, 0, 1, pool, None, None,
                                           s) == kvl.KVL_EINVAL
        for direction in (kvl.KVL_GATHER, kvl.KVL_SCATTER_BACK):
            assert kvl.kvl_gather_layer_objects(g, plan, small, reqs, tabs, 0, 1, pool, direction,
                                                None, s) == kvl.KVL_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(d.pool, before) and gb.status() == (0, 0)
    bad = kvl.geom(SPEC.L, SPEC.P, SPEC.B, 24, SPEC.n_pool)
    assert kvl.kvl_merge_scatter_paged(bad, plan, pb, reqs, tabs, 0, 1, pool, None, None, s) == kvl.KVL_EALIGN
    # launch options: a negative CTA cap, an unknown flag, both host flags
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, -1, s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, kvl.kvl_launch(4, 32),
                                       s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, kvl.kvl_launch(0, 3),
                                       s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, kvl.kvl_launch(0, 7),
                                       s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, kvl.kvl_launch(0, 64),
                                       s) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, reqs, tabs, 0, 1, pool, None, kvl.kvl_launch(0, 11),
                                       s) == kvl.KVL_EINVAL
    # a NULL request array is for plans of no requests: this plan refuses it on the device
    assert kvl.kvl_merge_scatter_paged(g, plan, pb, 0, tabs, 0, 1, pool, None, None, s) == kvl.KVL_OK
    assert gb.status()[0] == kvl.KVL_EINVAL
    gb.plan()
    assert gb.status() == (0, 0)
    # a plan built for another pool size is refused on the device
    other = kvl.geom(SPEC.L, SPEC.P, SPEC.B, SPEC.Rp, SPEC.n_pool - 1)
    assert kvl.kvl_merge_scatter_paged(other, plan, pb, reqs, tabs, 0, 1, pool, None, None, s) == kvl.KVL_OK
    assert gb.status()[0] == kvl.KVL_EINVAL
    # ... and so is one built for another row size or plane count (the boxes of its
    # tensor maps hold the plan's rows); the call copies nothing
    for other in (kvl.geom(SPEC.L, SPEC.P, SPEC.B, SPEC.Rp + 16, SPEC.n_pool),
                  kvl.geom(SPEC.L, 1, SPEC.B, SPEC.Rp, SPEC.n_pool)):
        gb.plan()
        assert gb.status() == (0, 0)
        before = d.pool.clone()
        assert kvl.kvl_merge_scatter_paged(other, plan, pb, reqs, tabs, 0, 1, pool, None, None,
                                           s) == kvl.KVL_OK
        assert kvl.kvl_slice_layer(other, plan, pb, reqs, 0, 1, pool, None, s) == kvl.KVL_OK
        assert gb.status()[0] == kvl.KVL_EINVAL
        assert torch.equal(d.pool, before)


def test_a_plan_holding_more_requests_than_the_stated_buffer_is_refused_on_the_device():
    """plan_bytes at least the geometry's smallest plan passes the host check, but the
    plan in the buffer records n_req requests whose sections end beyond plan_bytes: the
    kernels see that in the header, record KVL_EINVAL and read none of those sections;
    every buffer keeps its bytes.  The same plan with its full size then copies."""
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    gb.plan()
    g, plan, reqs, tabs = gb.g, gb.d_plan.data_ptr(), gb.d_reqs.data_ptr(), gb.tables.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    least, need = kvl.kvl_plan_layout(g, 0)[8], kvl.kvl_plan_layout(g, gb.n_req)[8]
    assert least < need <= gb.plan_bytes
    out = torch.full((gb.total_hit * SPEC.R + 64,), 0x3C, dtype=torch.uint8, device="cuda")
    pool0, obj0, out0 = d.pool.clone(), d.objects.clone(), out.clone()
    for short in (least, need - 16):
        gb.plan()
        assert kvl.kvl_slice_layer(g, plan, short, reqs, 0, 1, out.data_ptr(), None, s) == kvl.KVL_OK
        assert kvl.kvl_merge_scatter_paged(g, plan, short, reqs, tabs, 0, 1, d.pool.data_ptr(),
                                           None, None, s) == kvl.KVL_OK
        assert kvl.kvl_gather_layer_objects(g, plan, short, reqs, tabs, 0, 1, d.pool.data_ptr(),
                                            kvl.KVL_GATHER, None, s) == kvl.KVL_OK
        assert gb.status()[0] == kvl.KVL_EINVAL
        assert torch.equal(d.pool, pool0) and torch.equal(d.objects, obj0) and torch.equal(out, out0)
    gb.plan()
    assert kvl.kvl_merge_scatter_paged(g, plan, need, reqs, tabs, 0, 1, d.pool.data_ptr(), None,
                                       None, s) == kvl.KVL_OK
    ob = oracle.Batch(geom_of(SPEC), hb.layout.requests, hb.hit, hb.miss, hb.objects, hb.tables,
                      hb.src_tables)
    assert ob.merge_scatter(0, hb.pool)[0] == 0
    assert np.array_equal(d.pool.cpu().numpy(), hb.pool)
    assert gb.status() == (0, 0)


def test_a_wait_that_runs_out_reports_a_timeout_and_the_context_survives():
    """A bounded mbarrier wait whose bytes never arrive gives up after its limit and
    reports KVL_ETIMEOUT; the GPU stays usable for the copies that follow."""
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert kvl.kvl_diag_wait_timeout(20000, st.data_ptr(), s) == kvl.KVL_OK
    torch.cuda.synchronize()
    assert int(st.item()) == kvl.KVL_ETIMEOUT
    assert kvl.kvl_diag_wait_timeout(0, st.data_ptr(), s) == kvl.KVL_EINVAL
    # the context still works: a full parity round trip afterwards
    hb = host_buffers(SPEC)
    gb, d = device_batch(SPEC, hb)
    gb.plan()
    ob = oracle.Batch(geom_of(SPEC), hb.layout.requests, hb.hit, hb.miss, hb.objects,
                      hb.tables, hb.src_tables)
    for layer in range(SPEC.L):
        gb.merge_scatter(layer, d.pool)
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
    assert np.array_equal(d.pool.cpu().numpy(), hb.pool)
    assert gb.status() == (0, 0)
