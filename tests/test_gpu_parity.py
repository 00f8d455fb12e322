"""GPU parity: every kernel, through the C ABI, byte for byte against the CPU oracle.

Small cases (ragged batches that span many work items, mid-block hit/miss
boundaries, partial last blocks, permuted sources, both miss layouts, one and two
planes, row sizes from 16 B to 4 KiB, blocks of 1 to 64 tokens) compare whole
buffers, guard bytes included.  The full-size workloads run in the benchmark's
launch configuration and are compared with the oracle on sampled layers, with the
scatter-back round trip checked on every layer.
"""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._device import MappedHost, device_batch, mapped_copy, one_layer_problem, sentinel_dev
from tests._host import GUARD, geom_of, host_buffers

pytestmark = pytest.mark.gpu

SENT = workloads.SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    kvl.lib()


def oracle_batch(spec, hb):
    return oracle.Batch(geom_of(spec), hb.layout.requests, hb.hit, hb.miss, hb.objects,
                        hb.tables, hb.src_tables)


def assert_bytes_equal(got_t, want, what):
    got = got_t.cpu().numpy()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at {bad[0]}")


def run_parity(spec, *, check_injective=True, objects_one_layer=False, payload="bytes"):
    hb = host_buffers(spec, objects_one_layer=objects_one_layer)
    if payload == "spec":
        # the workload's own value distribution, made once on the CPU
        cpu = workloads.allocate(spec, "cpu", objects_one_layer=objects_one_layer)
        hb.hit[:cpu["hit"].numel()] = cpu["hit"].numpy()[:hb.hit.size]
        hb.miss[:cpu["miss"].numel()] = cpu["miss"].numpy()[:hb.miss.size]
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)

    gb.plan(check_injective=check_injective)
    op = ob.plan(check_injective=check_injective)
    gp = gb.plan_arrays()
    assert gb.status() == (0, 0) and op["status"] == 0
    for k in ("n_items", "tok_off", "hit_off", "blk_off", "item_req", "item_blk"):
        assert np.array_equal(np.asarray(gp[k]), np.asarray(op[k])), k

    R = spec.R
    hit_out = sentinel_dev(ob.total_hit() * R)
    complete = sentinel_dev(ob.total_tokens() * R)
    for layer in range(spec.L):
        gb.slice_layer(layer, hit_out)
        st, want_hit = ob.slice_layer(layer)
        assert st == 0
        assert_bytes_equal(hit_out[:want_hit.size], want_hit, f"hit_layer[{layer}]")
        assert torch.all(hit_out[want_hit.size:] == SENT)

        gb.merge_scatter(layer, d.pool, complete)
        st, want_comp = ob.merge_scatter(layer, hb.pool, want_complete=True)
        assert st == 0
        assert_bytes_equal(complete[:want_comp.size], want_comp, f"complete_layer[{layer}]")
        assert_bytes_equal(d.pool, hb.pool, f"pool after merge-scatter of layer {layer}")

        gb.gather(layer, d.pool)
        assert ob.gather_objects(layer, hb.pool) == 0
        assert_bytes_equal(d.objects, hb.objects, f"objects of layer {layer}")

    # scatter back into fresh pools, layer by layer
    d.pool.fill_(SENT)
    hb.pool[:] = SENT
    for layer in range(spec.L):
        if objects_one_layer:
            break
        gb.scatter_back(layer, d.pool)
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(d.pool, hb.pool, "pool after scatter-back")
    assert gb.status() == (0, 0)


def test_tiny_workload_bit_exact():
    run_parity(workloads.get_spec("tiny"), payload="spec")


RANDOM_CASES = 40


@pytest.mark.parametrize("case", range(RANDOM_CASES))
def test_random_ragged_batches_bit_exact(case):
    g = np.random.default_rng(9000 + case)
    P = int(g.integers(1, 3))
    Rp = int(g.choice([16, 48, 256, 1152, 2048]))
    B = int(g.choice([1, 3, 16, 64]))
    n = int(g.choice([1, 2, 7, 33]))
    max_t = int(max(8, min(1200, 400_000 // max(1, n * Rp * P))))
    t_hit = g.integers(0, max_t, n)
    t_miss = g.integers(0, max(2, max_t // 4), n)
    if case % 5 == 0:
        t_hit[0] = 0          # a miss-only request
    if case % 7 == 1 and n > 1:
        t_miss[-1] = 0        # a hit-only request
    spec = workloads.custom_spec(
        L=int(g.integers(1, 4)), P=P, B=B, Rp=Rp, t_hit=t_hit, t_miss=t_miss,
        table=str(g.choice(["perm", "fragmented", "identity"])),
        source=str(g.choice(["contiguous", "permuted"])),
        miss_order=str(g.choice(["layer", "token"])), seed=700 + case,
        objects=str(g.choice(["layer", "block"])))
    run_parity(spec)


MAPPED_CASES = 16


@pytest.mark.parametrize("case", range(MAPPED_CASES))
def test_random_ragged_batches_through_tensor_maps(case):
    """Ragged batches whose sources are large enough (a dim spanning 1 MiB or more)
    for the plan's tensor maps, so whole segments go through tiled tensor loads and
    the rest (hit/miss boundary blocks, partial last blocks, short segments) through
    per-row loads, side by side in one launch."""
    g = np.random.default_rng(9500 + case)
    P = int(g.integers(1, 3))
    Rp = int(g.choice([256, 1152, 2048, 4096]))
    B = int(g.choice([3, 16, 64]))
    L = int(g.integers(2, 5))
    n = int(g.choice([1, 3, 6]))
    R = P * Rp
    lo = -(-(1 << 20) // ((L - 1) * R)) + 1   # enough tokens for a 1 MiB hit span
    t_hit = g.integers(lo, 3 * lo, n)
    t_miss = g.integers(lo // 2, 2 * lo, n)
    if case % 4 == 0:
        t_miss[0] = int(g.integers(0, 3))   # hit blocks end inside a block
    spec = workloads.custom_spec(
        L=L, P=P, B=B, Rp=Rp, t_hit=t_hit, t_miss=t_miss,
        table=str(g.choice(["perm", "fragmented"])),
        source=str(g.choice(["contiguous", "permuted"])),
        miss_order=str(g.choice(["layer", "token"])), seed=950 + case,
        objects=str(g.choice(["layer", "block"])))
    hb = host_buffers(spec)
    gb, _ = device_batch(spec, hb)
    gb.plan()
    flags = gb.d_plan.cpu().numpy()[256:256 + 128 * gb.n_items].view(np.int32).reshape(-1, 32)[:, 29]
    assert (flags & 1).any() and (flags & 2).any(), "no hit maps were built"
    run_parity(spec)


def _mapped_spec(seed):
    """A random batch whose sources span a megabyte or more (tensor maps), over plane
    rows whose segments leave block tails (1,152, 1,536, 3,072 B ...), odd block
    sizes, permuted or contiguous sources, both miss layouts, empty hit prefixes."""
    g = np.random.default_rng(seed)
    P = int(g.integers(1, 3))
    Rp = int(g.choice([256, 1152, 1536, 2048, 3072, 4096, 8192]))
    if P * Rp > 32768:
        P = 1
    B = int(g.choice([3, 7, 16, 31, 64]))
    L = int(g.integers(2, 6))
    n = int(g.choice([1, 2, 4, 7]))
    lo = -(-(1 << 20) // ((L - 1) * P * Rp)) + 1
    t_hit = g.integers(lo // 2, 3 * lo, n)
    t_miss = g.integers(0, 2 * lo, n)
    if g.random() < 0.3:
        t_hit[0] = 0
    return g, workloads.custom_spec(
        f"mapped{seed}", L=L, P=P, B=B, Rp=Rp, t_hit=t_hit, t_miss=t_miss,
        table=str(g.choice(["perm", "fragmented"])),
        source=str(g.choice(["contiguous", "permuted"])),
        miss_order=str(g.choice(["layer", "token"])), seed=seed,
        objects=str(g.choice(["layer", "block"])))


@pytest.mark.parametrize("case", range(40))
def test_random_mapped_batches_with_tails(case):
    run_parity(_mapped_spec(96000 + case)[1])


TAIL_CASES = {
    # blocks whose rows do not divide into whole segments, so each block ends in a tail
    # read through the tail maps: 64-token blocks of 1,152-byte rows (28 + 28 + 8),
    # 3 KiB planes in 16-token blocks (10 + 6; slice rows of 6 KiB: 5 + 5 + 5 + 1),
    # 16 KiB planes in 3-token blocks (2 + 1)
    "latent_rows": dict(L=2, P=1, B=64, Rp=1152, t_hit=[1700, 900, 2500],
                        t_miss=[130, 2000, 7]),
    "3k_planes": dict(L=3, P=2, B=16, Rp=3072, t_hit=[600, 37], t_miss=[450, 200],
                      source="permuted"),
    "16k_planes": dict(L=2, P=2, B=3, Rp=16384, t_hit=[40, 25], t_miss=[17, 40],
                       miss_order="token"),
}


@pytest.mark.parametrize("name", sorted(TAIL_CASES))
def test_block_tails_through_tensor_maps(name):
    spec = workloads.custom_spec(name, **TAIL_CASES[name], table="perm", seed=61)
    hb = host_buffers(spec)
    gb, _ = device_batch(spec, hb)
    gb.plan()
    flags = gb.d_plan.cpu().numpy()[256:256 + 128 * gb.n_items].view(np.int32).reshape(-1, 32)[:, 29]
    assert (flags & (1 << 3)).any(), "no block-tail maps of the hit rows were built"
    run_parity(spec)


SCALED = {
    # the shapes of the four larger workloads, with fewer layers and tokens
    "llama3_8b_agentic": dict(L=3, P=2, B=16, Rp=2048, t_hit=[3000], t_miss=[77], table="perm"),
    "qwen3_32b_long": dict(L=2, P=2, B=64, Rp=2048, t_hit=[5000], t_miss=[1700], table="perm",
                           source="permuted"),
    "latent_batch": dict(L=2, P=1, B=64, Rp=1152, t_hit=[1700, 900, 2500, 64, 1300],
                         t_miss=[130, 2000, 7, 64, 1], table="perm"),
    "many_small": dict(L=2, P=2, B=16, Rp=2048, t_hit=list(range(37, 37 + 40 * 23, 23)),
                       t_miss=[16 + (7 * i) % 240 for i in range(40)], table="fragmented"),
}


@pytest.mark.parametrize("name", sorted(SCALED))
def test_scaled_workload_shapes_bit_exact(name):
    run_parity(workloads.custom_spec(name, **SCALED[name], seed=31))


EDGE = {
    # degenerate batches: no requests at all, only empty requests, empty requests
    # between others, a single token
    "no_requests": dict(L=2, P=2, B=16, Rp=256, t_hit=[], t_miss=[]),
    "only_empty_requests": dict(L=2, P=2, B=16, Rp=256, t_hit=[0, 0], t_miss=[0, 0]),
    "empty_requests_between": dict(L=3, P=2, B=16, Rp=64, t_hit=[0, 17, 0, 0], t_miss=[0, 0, 5, 0]),
    "one_token": dict(L=1, P=2, B=64, Rp=16, t_hit=[0], t_miss=[1]),
    # the largest rows a 32 KiB stage holds: a 32 KiB slice row (2 planes of 16 KiB)
    # and a 32 KiB plane row
    "largest_slice_row": dict(L=2, P=2, B=2, Rp=16384, t_hit=[3, 0, 1], t_miss=[2, 1, 0]),
    "largest_plane_row": dict(L=2, P=1, B=3, Rp=32768, t_hit=[4, 1], t_miss=[0, 3]),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_shapes_bit_exact(name):
    run_parity(workloads.custom_spec(**EDGE[name], source="permuted", seed=301))


def test_rows_larger_than_a_stage_are_refused():
    """A slice row of two 32 KiB planes does not fit a 32 KiB stage: the slice is refused
    on the host; the per-plane ops, whose rows are one plane, still run."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(L=1, P=2, B=2, Rp=32768, t_hit=[3], t_miss=[1], seed=302)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    out = sentinel_dev(ob.total_hit() * spec.R)
    s = torch.cuda.current_stream().cuda_stream
    assert kvl.kvl_slice_layer(gb.g, gb.d_plan.data_ptr(), gb.plan_bytes, gb.d_reqs.data_ptr(), 0, 1,
                               out.data_ptr(), None, s) == kvl.KVL_EINVAL
    gb.merge_scatter(0, d.pool)
    assert ob.merge_scatter(0, hb.pool)[0] == 0
    assert_bytes_equal(d.pool, hb.pool, "pool")
    assert gb.status() == (0, 0)


def test_without_injectivity_check_results_are_unchanged():
    spec = workloads.custom_spec(L=2, P=2, B=16, Rp=256, t_hit=[300, 5], t_miss=[20, 40])
    run_parity(spec, check_injective=False)


def test_block_major_object_files():
    spec = workloads.custom_spec(L=4, P=2, B=16, Rp=2048, t_hit=[700, 0, 130], t_miss=[33, 90, 0],
                                 source="permuted", objects="block", seed=77)
    run_parity(spec)


MULTI_LAYER_SPECS = {
    # sources far below a tensor map's span (every row its own load), and sources of
    # megabytes (whole segments through the maps, each unit at its own layer)
    "small_rows": dict(L=4, P=2, B=16, Rp=256, t_hit=[300, 0, 77, 41], t_miss=[20, 33, 0, 5]),
    "mapped_rows": dict(L=4, P=2, B=16, Rp=2048, t_hit=[700, 0, 300, 41],
                        t_miss=[400, 33, 0, 5]),
}


@pytest.mark.parametrize("rows", sorted(MULTI_LAYER_SPECS))
@pytest.mark.parametrize("layers", [(0, 4), (1, 2), (3, 1)])
def test_multi_layer_launches_equal_the_layer_by_layer_oracle(layers, rows):
    first, count = layers
    spec = workloads.custom_spec(rows, **MULTI_LAYER_SPECS[rows], source="permuted", seed=91,
                                 objects="block")
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    flags = gb.d_plan.cpu().numpy()[256:256 + 128 * gb.n_items].view(np.int32).reshape(-1, 32)[:, 29]
    assert bool((flags & 1).any()) == (rows == "mapped_rows")
    R = spec.R
    n_hit, n_tok = ob.total_hit() * R, ob.total_tokens() * R
    hit_out = sentinel_dev(count * n_hit)
    complete = sentinel_dev(count * n_tok)
    gb.slice_layer(first, hit_out, layer_count=count)
    gb.merge_scatter(first, d.pool, complete, layer_count=count)
    gb.gather(first, d.pool, layer_count=count)
    want_hit = np.full(count * n_hit + GUARD, SENT, np.uint8)
    want_comp = np.full(count * n_tok + GUARD, SENT, np.uint8)
    for i, layer in enumerate(range(first, first + count)):
        want_hit[i * n_hit:(i + 1) * n_hit] = ob.slice_layer(layer)[1]
        want_comp[i * n_tok:(i + 1) * n_tok] = ob.merge_scatter(layer, hb.pool, want_complete=True)[1]
        assert ob.gather_objects(layer, hb.pool) == 0
    assert_bytes_equal(hit_out, want_hit, "hit_out")
    assert_bytes_equal(complete, want_comp, "complete_out")
    assert_bytes_equal(d.pool, hb.pool, "pool")
    assert_bytes_equal(d.objects, hb.objects, "objects")
    d.pool.fill_(SENT)
    hb.pool[:] = SENT
    gb.scatter_back(first, d.pool, layer_count=count)
    for layer in range(first, first + count):
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(d.pool, hb.pool, "pool after scatter-back")
    assert gb.status() == (0, 0)


@pytest.mark.parametrize("max_ctas", [1, 3, 17])
def test_an_sm_budget_changes_nothing_but_speed(max_ctas):
    spec = workloads.custom_spec(L=2, P=2, B=16, Rp=512, t_hit=[900, 0, 77, 410],
                                 t_miss=[20, 133, 0, 5], source="permuted", seed=93)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    hit_out = sentinel_dev(ob.total_hit() * spec.R)
    for layer in range(spec.L):
        gb.slice_layer(layer, hit_out, max_ctas=max_ctas)
        gb.merge_scatter(layer, d.pool, max_ctas=max_ctas)
        gb.gather(layer, d.pool, max_ctas=max_ctas)
        want_hit = ob.slice_layer(layer)[1]
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
        assert ob.gather_objects(layer, hb.pool) == 0
        assert_bytes_equal(hit_out[:want_hit.size], want_hit, "hit_out")
        assert_bytes_equal(d.pool, hb.pool, "pool")
        assert_bytes_equal(d.objects, hb.objects, "objects")
    d.pool.fill_(SENT)
    hb.pool[:] = SENT
    for layer in range(spec.L):
        gb.scatter_back(layer, d.pool, max_ctas=max_ctas)
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(d.pool, hb.pool, "pool after scatter-back")
    assert gb.status() == (0, 0)


def _claim_counters(gb):
    """The plan's per-(layer, op) claim counters, [L][4] x (next, reserved)."""
    off = gb.layout[7]
    return gb.d_plan[off:off + gb.L * 4 * 8].cpu().numpy().view(np.uint32).reshape(gb.L, 4, 2)


# 26 work items per layer: the CTA caps below give fewer items than CTAs (whole GPU,
# 40), between one and two per CTA (20), exactly two (13) and more (5, 1), so the
# launch's count of claims, max(units - 2G, 0) + G, takes each of its forms.
@pytest.mark.parametrize("max_ctas", [None, 40, 20, 13, 5, 1])
@pytest.mark.parametrize("layer_count", [1, 2])
def test_repeated_launches_on_one_plan_rewind_their_claim_counters(max_ctas, layer_count):
    spec = workloads.custom_spec(L=3, P=2, B=16, Rp=512, t_hit=[300, 66], t_miss=[20, 30],
                                 source="contiguous", seed=71)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    assert gb.n_items == 26
    R, l0 = spec.R, 1
    n_hit = ob.total_hit() * R
    want_hit = np.concatenate([ob.slice_layer(l)[1] for l in range(l0, l0 + layer_count)])
    for l in range(l0, l0 + layer_count):
        assert ob.merge_scatter(l, hb.pool)[0] == 0
        assert ob.gather_objects(l, hb.pool) == 0
    pool_want, obj_want = hb.pool.copy(), hb.objects.copy()
    pool0 = d.pool.clone()
    for rep in range(3):
        # each launch starts from a fresh destination, so every byte is this launch's
        hit_out = sentinel_dev(layer_count * n_hit)
        gb.slice_layer(l0, hit_out, layer_count=layer_count, max_ctas=max_ctas)
        assert_bytes_equal(hit_out[:want_hit.size], want_hit, f"hit_out, launch {rep}")
        assert not _claim_counters(gb).any(), f"counters after slice launch {rep}"
        d.pool.copy_(pool0)
        gb.merge_scatter(l0, d.pool, layer_count=layer_count, max_ctas=max_ctas)
        d.objects.fill_(SENT)
        gb.gather(l0, d.pool, layer_count=layer_count, max_ctas=max_ctas)
        assert_bytes_equal(d.pool, pool_want, f"pool, launch {rep}")
        assert_bytes_equal(d.objects, obj_want, f"objects, launch {rep}")
        assert not _claim_counters(gb).any(), f"counters after merge and gather {rep}"
        d.pool.fill_(SENT)
        gb.scatter_back(l0, d.pool, layer_count=layer_count, max_ctas=max_ctas)
        back = hb.pool.copy()
        back[:] = SENT
        for l in range(l0, l0 + layer_count):
            assert ob.scatter_back(l, back) == 0
        assert_bytes_equal(d.pool, back, f"pool after scatter-back, launch {rep}")
        assert not _claim_counters(gb).any(), f"counters after scatter-back {rep}"
    assert gb.status() == (0, 0)


@pytest.mark.parametrize("budgets", [(None,), (5, None, 2, 11)])
def test_overlapped_layer_launches_equal_the_oracle(budgets):
    """Each op's launches for successive layers carry KVL_LAUNCH_OVERLAP_PREVIOUS (all
    but the first of each phase): a launch may start while the one before it runs,
    and a phase's first launch, which reads the previous phase's output, must still
    see every earlier launch complete.  Mixed SM budgets let several launches of a
    chain run at once."""
    import layer_wise_paged_gb300 as kvl
    ov = kvl.KVL_LAUNCH_OVERLAP_PREVIOUS
    spec = workloads.custom_spec(L=8, P=2, B=16, Rp=1024, t_hit=[3000, 0, 777, 1410],
                                 t_miss=[200, 1333, 0, 55], source="permuted", seed=97)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    R = spec.R
    n_hit, n_tok = ob.total_hit() * R, ob.total_tokens() * R
    hit_out = sentinel_dev(spec.L * n_hit)
    complete = sentinel_dev(spec.L * n_tok)

    def opts(layer):
        return dict(max_ctas=budgets[layer % len(budgets)],
                    flags=ov if layer else kvl.KVL_LAUNCH_SHARE_SMS * (len(budgets) > 1))

    for layer in range(spec.L):
        gb.slice_layer(layer, hit_out[layer * n_hit:], **opts(layer))
    for layer in range(spec.L):
        gb.merge_scatter(layer, d.pool, complete[layer * n_tok:], **opts(layer))
    for layer in range(spec.L):
        gb.gather(layer, d.pool, **opts(layer))
    want_hit = np.full(spec.L * n_hit + GUARD, SENT, np.uint8)
    want_comp = np.full(spec.L * n_tok + GUARD, SENT, np.uint8)
    for layer in range(spec.L):
        want_hit[layer * n_hit:(layer + 1) * n_hit] = ob.slice_layer(layer)[1]
        want_comp[layer * n_tok:(layer + 1) * n_tok] = ob.merge_scatter(
            layer, hb.pool, want_complete=True)[1]
        assert ob.gather_objects(layer, hb.pool) == 0
    assert_bytes_equal(hit_out, want_hit, "hit_out")
    assert_bytes_equal(complete, want_comp, "complete_out")
    assert_bytes_equal(d.pool, hb.pool, "pool")
    assert_bytes_equal(d.objects, hb.objects, "objects")
    d.pool.fill_(SENT)
    hb.pool[:] = SENT
    for layer in range(spec.L):
        gb.scatter_back(layer, d.pool, **opts(layer))
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(d.pool, hb.pool, "pool after scatter-back")
    assert gb.status() == (0, 0)


HOST_SPEC = dict(L=2, P=2, B=16, Rp=512, t_hit=[900, 0, 77, 410], t_miss=[20, 133, 0, 5],
                 source="permuted", seed=95)


def _host_batch(spec, hb, *, hit_host=False, miss_host=False, objects_host=False):
    """A GPU batch whose chosen buffers live in pinned, mapped host memory."""
    from layer_wise_paged_gb300.batch import Batch
    from tests._device import to_dev
    hit = mapped_copy(hb.hit) if hit_host else to_dev(hb.hit)
    miss = mapped_copy(hb.miss) if miss_host else to_dev(hb.miss)
    objects = mapped_copy(hb.objects) if objects_host else to_dev(hb.objects)
    tables, src_tables, pool = to_dev(hb.tables), to_dev(hb.src_tables), to_dev(hb.pool)
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    b = Batch(g, hb.layout.requests, hit, miss, objects, tables, src_tables)
    return b, hit, miss, objects, pool


def test_merge_scatter_and_slice_read_a_host_full_block():
    """DualPath's host buffer -> HBM leg: hit and miss rows read from pinned Grace
    memory, written to the HBM pool and hit_layer."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(**HOST_SPEC)
    hb = host_buffers(spec)
    gb, hit, miss, objects, pool = _host_batch(spec, hb, hit_host=True, miss_host=True)
    ob = oracle_batch(spec, hb)
    gb.plan()
    hit_out = sentinel_dev(ob.total_hit() * spec.R)
    for layer in range(spec.L):
        gb.slice_layer(layer, hit_out, flags=kvl.KVL_LAUNCH_HOST_SRC)
        gb.merge_scatter(layer, pool, flags=kvl.KVL_LAUNCH_HOST_SRC)
        want_hit = ob.slice_layer(layer)[1]
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
        assert_bytes_equal(hit_out[:want_hit.size], want_hit, "hit_out")
        assert_bytes_equal(pool, hb.pool, "pool")
    # all layers in one launch as well (the final H2D of the whole prompt KV)
    pool.fill_(SENT)
    gb.merge_scatter(0, pool, layer_count=spec.L, flags=kvl.KVL_LAUNCH_HOST_SRC)
    assert_bytes_equal(pool, hb.pool, "pool, one launch")
    assert gb.status() == (0, 0)


def test_host_memory_launches_ignore_plan_ready():
    """KVL_LAUNCH_PLAN_READY is accepted beside the host-memory flags and changes
    nothing there: their launches read or write host memory with SM loads or stores
    and keep the plain wait."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(**HOST_SPEC)
    hb = host_buffers(spec)
    gb, hit, miss, objects, pool = _host_batch(spec, hb, hit_host=True, miss_host=True)
    ob = oracle_batch(spec, hb)
    gb.plan()
    for layer in range(spec.L):
        f = kvl.KVL_LAUNCH_HOST_SRC | (kvl.KVL_LAUNCH_PLAN_READY if layer else 0)
        gb.merge_scatter(layer, pool, flags=f)
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
    assert_bytes_equal(pool, hb.pool, "pool")
    assert gb.status() == (0, 0)


def test_gather_writes_host_objects_and_scatter_back_reads_them():
    """Objects ready for transfer land in pinned host memory, and are restored from it."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(**HOST_SPEC, objects="block")
    hb = host_buffers(spec)
    gb, hit, miss, objects, pool = _host_batch(spec, hb, objects_host=True)
    ob = oracle_batch(spec, hb)
    gb.plan()
    complete = MappedHost(ob.total_tokens() * spec.R + GUARD)
    complete.np[:] = SENT
    for layer in range(spec.L):
        gb.merge_scatter(layer, pool, complete, flags=kvl.KVL_LAUNCH_HOST_DST)
        gb.gather(layer, pool, flags=kvl.KVL_LAUNCH_HOST_DST)
        torch.cuda.synchronize()
        want_comp = ob.merge_scatter(layer, hb.pool, want_complete=True)[1]
        assert ob.gather_objects(layer, hb.pool) == 0
        assert np.array_equal(complete.np[:want_comp.size], want_comp)
        assert np.all(complete.np[want_comp.size:] == SENT)
        assert_bytes_equal(pool, hb.pool, "pool")
        assert np.array_equal(objects.np[:hb.objects.size], hb.objects)
    pool.fill_(SENT)
    hb.pool[:] = SENT
    gb.scatter_back(0, pool, layer_count=spec.L, flags=kvl.KVL_LAUNCH_HOST_SRC)
    for layer in range(spec.L):
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(pool, hb.pool, "pool after scatter-back from host")
    assert gb.status() == (0, 0)


@pytest.mark.parametrize("rows", [2048, 1152])
def test_plan_ready_launches_read_what_the_kernel_before_them_writes(rows):
    """Every launch after the first carries KVL_LAUNCH_PLAN_READY and reads what the
    launch just before it writes: merge-scatter of layer l, then the gather of that
    layer's blocks, then their scatter-back into a second pool, layer after layer, with
    the slice of the next layer between (a lone launch of another op).  Each waiting
    launch prefetches its first rows into L2 while its predecessor still writes them;
    the results must still be the oracle's, byte for byte."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(L=4, P=2 if rows == 2048 else 1, B=16, Rp=rows,
                                 t_hit=[2100, 700, 1500], t_miss=[90, 400, 33],
                                 table="fragmented", source="permuted", seed=8801 + rows)
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    R, L = spec.R, spec.L
    n_hit = ob.total_hit() * R
    hit_out = sentinel_dev(L * n_hit)
    pool2 = torch.full_like(d.pool, SENT)
    ready = kvl.KVL_LAUNCH_PLAN_READY
    for layer in range(L):
        gb.slice_layer(layer, hit_out[layer * n_hit:], flags=ready if layer else 0)
        gb.merge_scatter(layer, d.pool, flags=ready)
        gb.gather(layer, d.pool, flags=ready)
        gb.scatter_back(layer, pool2, flags=ready, max_ctas=[None, 7][layer % 2])
    want_hit = np.full(L * n_hit + GUARD, SENT, np.uint8)
    pool2_h = np.full_like(hb.pool, SENT)
    for layer in range(L):
        want_hit[layer * n_hit:(layer + 1) * n_hit] = ob.slice_layer(layer)[1]
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
        assert ob.gather_objects(layer, hb.pool) == 0
        assert ob.scatter_back(layer, pool2_h) == 0
    assert_bytes_equal(hit_out, want_hit, "hit_out")
    assert_bytes_equal(d.pool, hb.pool, "pool")
    assert_bytes_equal(d.objects, hb.objects, "objects")
    assert_bytes_equal(pool2, pool2_h, "second pool")
    assert gb.status() == (0, 0)


@pytest.mark.parametrize("case", range(46))
def test_random_launch_plans_equal_the_oracle(case):
    """Random ragged batches under random launch plans: per op, random layers per
    launch, SM budgets and overlap flags (every launch of a phase after the first may
    overlap its predecessor; the first shares SMs or not), and KVL_LAUNCH_PLAN_READY on
    any launch but the first after the plan (a phase's first launch then prefetches the
    rows the phase before it is still writing).  Budgets as small as one CTA let long
    chains of launches run at once.  Cases 30 and up draw batches large enough for
    tensor maps."""
    import layer_wise_paged_gb300 as kvl
    if case >= 30:
        g, spec = _mapped_spec(97000 + case)
        L = spec.L
    else:
        g = np.random.default_rng(7100 + case)
        L = int(g.integers(2, 7))
        n = int(g.choice([1, 3, 9]))
        spec = workloads.custom_spec(
            L=L, P=int(g.integers(1, 3)), B=int(g.choice([4, 16, 64])),
            Rp=int(g.choice([64, 1152, 2048])), t_hit=g.integers(0, 900, n),
            t_miss=g.integers(0, 300, n), table=str(g.choice(["perm", "fragmented"])),
            source=str(g.choice(["contiguous", "permuted"])), seed=7200 + case,
            objects=str(g.choice(["layer", "block"])))
    hb = host_buffers(spec)
    gb, d = device_batch(spec, hb)
    ob = oracle_batch(spec, hb)
    gb.plan()
    R = spec.R
    n_hit, n_tok = ob.total_hit() * R, ob.total_tokens() * R
    hit_out = sentinel_dev(L * n_hit)
    complete = sentinel_dev(L * n_tok)

    def plan_of_launches(after_plan=False):
        K = int(g.integers(1, L + 1))
        out = []
        for i, l0 in enumerate(range(0, L, K)):
            f = 0
            if i == 0 and g.random() < 0.5:
                f = kvl.KVL_LAUNCH_SHARE_SMS
            elif i > 0 and g.random() < 0.8:
                f = kvl.KVL_LAUNCH_OVERLAP_PREVIOUS
            if not (after_plan and i == 0) and g.random() < 0.7:
                f |= kvl.KVL_LAUNCH_PLAN_READY
            out.append((l0, min(K, L - l0), dict(max_ctas=[None, 1, 5, 40][int(g.integers(0, 4))],
                                                  flags=f)))
        return out

    for l0, k, o in plan_of_launches(after_plan=True):
        gb.slice_layer(l0, hit_out[l0 * n_hit:], layer_count=k, **o)
    for l0, k, o in plan_of_launches():
        gb.merge_scatter(l0, d.pool, complete[l0 * n_tok:], layer_count=k, **o)
    for l0, k, o in plan_of_launches():
        gb.gather(l0, d.pool, layer_count=k, **o)
    want_hit = np.full(L * n_hit + GUARD, SENT, np.uint8)
    want_comp = np.full(L * n_tok + GUARD, SENT, np.uint8)
    for layer in range(L):
        want_hit[layer * n_hit:(layer + 1) * n_hit] = ob.slice_layer(layer)[1]
        want_comp[layer * n_tok:(layer + 1) * n_tok] = ob.merge_scatter(
            layer, hb.pool, want_complete=True)[1]
        assert ob.gather_objects(layer, hb.pool) == 0
    assert_bytes_equal(hit_out, want_hit, "hit_out")
    assert_bytes_equal(complete, want_comp, "complete_out")
    assert_bytes_equal(d.pool, hb.pool, "pool")
    assert_bytes_equal(d.objects, hb.objects, "objects")
    d.pool.fill_(SENT)
    hb.pool[:] = SENT
    for l0, k, o in plan_of_launches():
        gb.scatter_back(l0, d.pool, layer_count=k, **o)
    for layer in range(L):
        assert ob.scatter_back(layer, hb.pool) == 0
    assert_bytes_equal(d.pool, hb.pool, "pool after scatter-back")
    assert gb.status() == (0, 0)


def test_host_legs_with_overlapped_launches():
    """The host-memory variants honour KVL_LAUNCH_OVERLAP_PREVIOUS too: successive
    layers read from a pinned host full block, each launch overlapping the one before."""
    import layer_wise_paged_gb300 as kvl
    spec = workloads.custom_spec(**dict(HOST_SPEC, L=4))
    hb = host_buffers(spec)
    gb, hit, miss, objects, pool = _host_batch(spec, hb, hit_host=True, miss_host=True)
    ob = oracle_batch(spec, hb)
    gb.plan()
    n_hit = ob.total_hit() * spec.R
    hit_out = sentinel_dev(spec.L * n_hit)
    src = kvl.KVL_LAUNCH_HOST_SRC
    for layer in range(spec.L):
        gb.slice_layer(layer, hit_out[layer * n_hit:],
                       flags=src | (kvl.KVL_LAUNCH_OVERLAP_PREVIOUS if layer else 0))
    for layer in range(spec.L):
        gb.merge_scatter(layer, pool, flags=src | (kvl.KVL_LAUNCH_OVERLAP_PREVIOUS if layer else 0))
    want_hit = np.full(spec.L * n_hit + GUARD, SENT, np.uint8)
    for layer in range(spec.L):
        want_hit[layer * n_hit:(layer + 1) * n_hit] = ob.slice_layer(layer)[1]
        assert ob.merge_scatter(layer, hb.pool)[0] == 0
    assert_bytes_equal(hit_out, want_hit, "hit_out")
    assert_bytes_equal(pool, hb.pool, "pool")
    assert gb.status() == (0, 0)


def test_objects_with_zero_layer_stride():
    spec = workloads.custom_spec(L=3, P=2, B=16, Rp=256, t_hit=[100, 50], t_miss=[3, 60])
    run_parity(spec, objects_one_layer=True)


# --------------------------------------------------------------------------
# Full-size workloads, sampled layers
# --------------------------------------------------------------------------

FULL = ["llama3_8b_agentic", "qwen3_32b_long", "latent_batch", "many_small"]


def _free_gb():
    # free to the driver plus free inside torch's cache
    free, _ = torch.cuda.mem_get_info()
    return (free + torch.cuda.memory_reserved() - torch.cuda.memory_allocated()) / 1e9


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled_layers(name):
    from layer_wise_paged_gb300.batch import Batch
    spec = workloads.get_spec(name)
    one_layer = name in ("latent_batch", "many_small", "qwen3_32b_long")
    need = workloads.footprint_bytes(spec, objects_one_layer=one_layer) / 1e9
    if need + 8 > _free_gb():
        pytest.skip(f"{name} needs {need:.0f} GB of device memory")
    bufs = workloads.allocate(spec, "cuda", objects_one_layer=one_layer)
    lay = bufs["layout"]
    g = (spec.L, spec.P, spec.B, spec.Rp, spec.n_pool)
    gb = Batch(g, lay.requests, bufs["hit"], bufs["miss"], bufs["objects"], bufs["tables"],
               bufs["src_tables"])
    gb.plan()
    assert gb.status() == (0, 0)
    R, layer_bytes = spec.R, spec.P * spec.n_pool * spec.B * spec.Rp
    pool = bufs["pool"]
    hit_out = sentinel_dev(gb.total_hit * R)
    sampled = {0, spec.L // 2, spec.L - 1}
    for layer in range(spec.L):
        region = pool[layer * layer_bytes:(layer + 1) * layer_bytes]
        before = region.cpu().numpy() if layer in sampled else None
        gb.slice_layer(layer, hit_out)
        gb.merge_scatter(layer, pool)
        gb.gather(layer, pool)
        # round trip on every layer: scatter-back into a blanked layer restores it
        after = region.clone()
        region.fill_(SENT)
        gb.scatter_back(layer, pool)
        assert torch.equal(region, after), f"{name}: scatter-back round trip, layer {layer}"
        del after
        if layer in sampled:
            dev = SimpleNamespace(hit=bufs["hit"], miss=bufs["miss"], tables=bufs["tables"],
                                  src_tables=bufs["src_tables"])
            ob, objs, obj_offs, host_pool = one_layer_problem(spec, lay, dev, layer, before)
            st, want_hit = ob.slice_layer(0)
            assert st == 0
            assert_bytes_equal(hit_out[:want_hit.size], want_hit, f"{name} hit_layer[{layer}]")
            assert ob.merge_scatter(0, host_pool)[0] == 0
            assert_bytes_equal(region, host_pool, f"{name} pool layer {layer}")
            assert ob.gather_objects(0, host_pool) == 0
            for q, o in zip(lay.requests, obj_offs):
                nb = spec.P * (-(-(q.t_hit + q.t_miss) // spec.B)) * spec.B * spec.Rp
                a = q.obj_off + layer * q.obj_layer_stride
                assert_bytes_equal(bufs["objects"][a:a + nb], objs[o:o + nb],
                                   f"{name} objects layer {layer}")
    assert gb.status() == (0, 0)
    del bufs, gb, pool, hit_out
    torch.cuda.empty_cache()
