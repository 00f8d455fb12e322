"""The C ABI without a GPU: the library builds, loads and exports every entry point
include/kvl.h declares; the binding's structs match the header's; host-side
argument checks answer before anything touches the device."""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

import layer_wise_paged_gb300 as kvl

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "kvl.h"


@pytest.fixture(scope="module")
def lib():
    kvl.build()
    return kvl.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(kvl_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", str(kvl.LIB)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (kvl_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_struct_layouts_match_the_header(tmp_path):
    prog = tmp_path / "layout.c"
    fields = [f for f in kvl.REQUEST_DTYPE.names]
    body = "\n".join(f'printf("{f} %zu\\n", offsetof(kvl_request, {f}));' for f in fields)
    prog.write_text(f"""
#include <stdio.h>
#include <stddef.h>
#include "kvl.h"
int main(void) {{
  printf("sizeof_request %zu\\n", sizeof(kvl_request));
  printf("sizeof_geom %zu\\n", sizeof(kvl_geom));
  printf("geom_pool_blocks %zu\\n", offsetof(kvl_geom, pool_blocks));
  {body}
  return 0;
}}""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", str(ROOT / "include"), str(prog), "-o", str(exe)],
                   check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                          text=True, check=True).stdout.splitlines())
    assert int(got["sizeof_request"]) == kvl.REQUEST_DTYPE.itemsize == 112
    assert int(got["sizeof_geom"]) == ctypes.sizeof(kvl.kvl_geom)
    assert int(got["geom_pool_blocks"]) == kvl.kvl_geom.pool_blocks.offset
    for f in fields:
        assert int(got[f]) == kvl.REQUEST_DTYPE.fields[f][1], f


def test_header_constants_match_the_binding():
    """Every #define KVL_<NAME> <integer> of the header has the same value in the binding."""
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    defines = {}
    for m in re.finditer(r"#define[ \t]+(KVL_[A-Z_]+)[ \t]+(\S.*)", text):
        expr = m.group(2).strip()
        assert re.fullmatch(r"[0-9x()<< ]+", expr), (m.group(1), expr)
        defines[m.group(1)] = eval(expr, {"__builtins__": {}})  # digits, shifts, parentheses
    assert {"KVL_OK", "KVL_ETIMEOUT", "KVL_LAUNCH_OVERLAP_PREVIOUS", "KVL_LAUNCH_SHARE_SMS",
            "KVL_STATIC_SCRATCH_POOL_BLOCKS"} <= set(defines)
    for name, value in defines.items():
        assert getattr(kvl, name) == value, name


def test_plan_layout_is_consistent(lib):
    for L, n, N in [(1, 0, 1), (2, 1, 32), (61, 16, 10625), (32, 256, 49262), (80, 1000, 1 << 20)]:
        g = kvl.geom(L, 2, 16, 256, N)
        off = kvl.kvl_plan_layout(g, n)
        assert off[0] == 0 and off[6] == 256  # records right after the 256-byte header
        assert all(o % 256 == 0 for o in off)
        need = {1: 8 * (n + 1), 2: 8 * (n + 1), 3: 8 * (n + 1), 4: 4 * N, 5: 4 * N,
                6: 128 * N, 7: 8 * 4 * L, 8: 4 * ((N + 31) // 32),
                10: (6 * 128 + 4) * n + 128}  # tensor maps (128-byte aligned), map flags
        starts = sorted((off[k], k) for k in need)
        ends = [s for s, _ in starts[1:]] + [off[9]]
        assert starts[0][0] >= 256
        for (start, k), end in zip(starts, ends):
            assert end - start >= need[k], k   # each section fits before the next one
        assert starts[-1][1] == 8              # the bitmap is the last section
        assert kvl.kvl_plan_bytes(g, n) == off[9]
    assert kvl.kvl_plan_bytes(kvl.geom(0, 2, 16, 256, 8), 1) == 0


def test_status_strings_and_launch_counts(lib):
    for c in range(7):
        assert kvl.kvl_status_string(c)
    assert kvl.kvl_launches_per_call(0) == 2
    assert [kvl.kvl_launches_per_call(w) for w in (1, 2, 3)] == [1, 1, 1]


def test_host_checks_answer_before_any_device_work(lib):
    good = kvl.geom(2, 2, 16, 256, 64)
    fake = 1 << 20  # never dereferenced: every call below fails its host checks first
    assert kvl.kvl_batch_plan(kvl.geom(0, 2, 16, 256, 64), 1, fake, fake, 1, fake, 1 << 20) == kvl.KVL_EINVAL
    assert kvl.kvl_batch_plan(kvl.geom(2, 2, 16, 24, 64), 1, fake, fake, 1, fake, 1 << 20) == kvl.KVL_EALIGN
    assert kvl.kvl_batch_plan(good, 1, fake, fake, 1, 0, 1 << 20) == kvl.KVL_EINVAL
    assert kvl.kvl_batch_plan(good, 1, fake, fake, 1, fake + 8, 1 << 20) == kvl.KVL_EALIGN
    assert kvl.kvl_batch_plan(good, 1, fake, fake, 1, fake, 16) == kvl.KVL_EINVAL
    assert kvl.kvl_batch_plan(good, -1, fake, fake, 1, fake, 1 << 20) == kvl.KVL_EINVAL
    pb = kvl.kvl_plan_bytes(good, 1)
    assert kvl.kvl_merge_scatter_paged(good, fake, pb, fake, fake, 2, 1, fake) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(good, fake, pb, fake, fake, 0, 1, fake + 4) == kvl.KVL_EALIGN
    assert kvl.kvl_merge_scatter_paged(good, fake, pb, fake, fake, 0, 0, fake) == kvl.KVL_EINVAL
    assert kvl.kvl_merge_scatter_paged(good, fake, pb, fake, fake, 1, 2, fake) == kvl.KVL_EINVAL
    assert kvl.kvl_gather_layer_objects(good, fake, pb, fake, fake, 0, 1, fake, 7) == kvl.KVL_EINVAL
    assert kvl.kvl_slice_layer(good, fake, pb, fake, 0, 1, 0) == kvl.KVL_EINVAL
    assert kvl.lib().kvl_read_status(None, None, None, None) == kvl.KVL_EINVAL


def test_copy_calls_refuse_a_plan_smaller_than_the_geometry_needs(lib):
    """A copy call is told the plan buffer's size; below the smallest plan of the
    geometry (kvl_plan_layout(geom, 0)[8]: header, one record per pool block, work
    list and counters) it returns KVL_EINVAL on the host, before any launch, for every
    op; at exactly that size the host lets it through to its remaining checks."""
    g = kvl.geom(2, 2, 16, 256, 64)
    fake = 1 << 20  # never dereferenced: each call below is refused on the host
    least = kvl.kvl_plan_layout(g, 0)[8]
    assert least < kvl.kvl_plan_layout(g, 5)[8]  # a plan of requests needs more
    assert least >= 256 + 128 * 64  # covers every item record a copy CTA reads first
    for pb in (0, 16, 256, least - 1):
        assert kvl.kvl_slice_layer(g, fake, pb, fake, 0, 1, fake) == kvl.KVL_EINVAL
        assert kvl.kvl_merge_scatter_paged(g, fake, pb, fake, fake, 0, 1, fake) == kvl.KVL_EINVAL
        for direction in (kvl.KVL_GATHER, kvl.KVL_SCATTER_BACK):
            assert kvl.kvl_gather_layer_objects(g, fake, pb, fake, fake, 0, 1, fake,
                                                direction) == kvl.KVL_EINVAL
    # at the least size the size check passes: a misaligned pool is what answers now
    assert kvl.kvl_merge_scatter_paged(g, fake, least, fake, fake, 0, 1, fake + 4) == kvl.KVL_EALIGN
    assert kvl.kvl_merge_scatter_paged(g, fake, least - 1, fake, fake, 0, 1, fake + 4) == kvl.KVL_EINVAL


def test_unit_numbering_limits_are_refused_on_the_host(lib):
    """Block ids are int32 and a launch numbers its (layer, item) units in 32 bits: a
    geometry with more than INT32_MAX pool blocks is refused by every call, and a copy
    call whose pool_blocks x layer_count reaches 2^31 returns KVL_EINVAL before any
    launch; one layer fewer passes that check (a misaligned pool answers instead)."""
    fake = 1 << 20  # never dereferenced: each call below is refused on the host
    too_many = kvl.geom(4, 2, 16, 256, (1 << 31))
    assert kvl.kvl_plan_bytes(too_many, 1) == 0
    assert kvl.kvl_merge_scatter_paged(too_many, fake, 1 << 62, fake, fake, 0, 1, fake) == kvl.KVL_EINVAL
    g = kvl.geom(4, 2, 16, 256, 1 << 30)
    least = kvl.kvl_plan_layout(g, 0)[8]
    for call in (lambda lc, pool: kvl.kvl_merge_scatter_paged(g, fake, least, fake, fake, 0, lc, pool),
                 lambda lc, pool: kvl.kvl_gather_layer_objects(g, fake, least, fake, fake, 0, lc, pool,
                                                               kvl.KVL_GATHER)):
        assert call(2, fake) == kvl.KVL_EINVAL      # 2^30 blocks x 2 layers = 2^31 units
        assert call(1, fake + 4) == kvl.KVL_EALIGN  # 2^30 units: on to the pool's alignment
    assert kvl.kvl_slice_layer(g, fake, least, fake, 1, 2, fake) == kvl.KVL_EINVAL
    assert kvl.kvl_slice_layer(g, fake, least, fake, 1, 1, fake + 4) == kvl.KVL_EALIGN


def test_request_packing_follows_layouts():
    import workloads
    spec = workloads.custom_spec(L=3, P=2, B=4, Rp=32, t_hit=[10, 0], t_miss=[3, 5],
                                 source="permuted")
    lay = workloads.layout(spec)
    arr = kvl.pack_requests(lay.requests, hit_base=1 << 32, miss_base=2 << 32,
                            obj_base=3 << 32, src_table_base=4 << 32)
    assert arr.shape == (2,)
    assert arr[0]["hit_src"] == (1 << 32) + lay.requests[0].hit_off
    assert arr[1]["hit_src"] == 0  # no hit tokens -> NULL
    assert arr[0]["hit_src_table"] == (4 << 32)
    assert arr[1]["miss_src"] == (2 << 32) + lay.requests[1].miss_off
    assert arr[1]["t_miss"] == 5 and arr[0]["t_hit"] == 10
