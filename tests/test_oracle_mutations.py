"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Every mutation is a one-line edit of ``oracle/kvl_oracle.c`` (a dropped term, a wrong
index or sign, a swapped operand) compiled into a separate library in a temporary
directory; the pin tests of ``test_oracle_pins.py`` then run against that library and
at least one of them must fail.  All mutations keep every access in bounds.
"""
from __future__ import annotations

import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTATIONS = {
    "miss_rows_overwrite_hit_rows": (
        "memcpy(complete_out + (row0 + q->t_hit + m) * R",
        "memcpy(complete_out + (row0 + m) * R"),
    "slot_off_by_one": (
        "pool_slot(g, pool, layer, p, b, t % g->B)",
        "pool_slot(g, pool, layer, p, b, (t + 1) % g->B)"),
    "planes_swapped": (
        "complete_layer + (row0 + t) * R + (int64_t)p * g->Rp",
        "complete_layer + (row0 + t) * R + (int64_t)(g->P - 1 - p) * g->Rp"),
    "layer_term_dropped": (
        "         + (int64_t)l * q->hit_layer_stride;", ";"),
    "blocks_floor_not_ceil": (
        "blk_off[r + 1] = blk_off[r] + ceil_div(th + tm, B);",
        "blk_off[r + 1] = blk_off[r] + (th + tm) / B;"),
    "gather_ignores_request_table_offset": (
        "int64_t b = tables[tab0 + j];", "int64_t b = tables[j];"),
    "object_plane_term_dropped": (
        "+ (int64_t)p * q->obj_plane_stride + j * q->obj_block_stride;",
        "+ j * q->obj_block_stride;"),
    "source_table_ignored": (
        "int64_t blk = q->hit_src_table ? q->hit_src_table[j] : j;",
        "int64_t blk = j;"),
    "miss_layer_term_dropped": (
        "return q->miss_src + t_miss_idx * q->miss_token_stride + (int64_t)l * q->miss_layer_stride;",
        "return q->miss_src + t_miss_idx * q->miss_token_stride;"),
    "scatter_table_offset_floor": (
        "        row0 += ta;\n        tab0 += ceil_div(ta, g->B);",
        "        row0 += ta;\n        tab0 += ta / g->B;"),
    "duplicate_not_flagged": (
        "if (seen[b]) {", "if (0) {"),
    "hit_prefix_sum_includes_miss": (
        "hit_off[r + 1] = hit_off[r] + th;", "hit_off[r + 1] = hit_off[r] + th + tm;"),
    "hit_slot_term_dropped": (
        "return q->hit_src + blk * q->hit_block_stride + s * q->hit_token_stride",
        "return q->hit_src + blk * q->hit_block_stride"),
    "hit_rows_of_previous_request": (
        "memcpy(complete_out + (row0 + t) * R, hit_layer + (hit0 + t) * R, (size_t)R);",
        "memcpy(complete_out + (row0 + t) * R, hit_layer + t * R, (size_t)R);"),
    "gather_reads_layer_zero": (
        "memcpy(obj, pool_slot(g, (uint8_t *)pool, layer, p, b, 0), (size_t)obj_bytes);",
        "memcpy(obj, pool_slot(g, (uint8_t *)pool, 0, p, b, 0), (size_t)obj_bytes);"),
    "scatter_uses_block_index_not_table": (
        "int64_t b = tables[tab0 + t / g->B];", "int64_t b = (tab0 + t / g->B) % g->n_pool;"),
    "gather_object_layer_term_dropped": (
        "uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride",
        "uint8_t *obj = q->objects + 0 * q->obj_layer_stride"),
    "gather_copies_one_row_of_a_block": (
        "memcpy(obj, pool_slot(g, (uint8_t *)pool, layer, p, b, 0), (size_t)obj_bytes);",
        "memcpy(obj, pool_slot(g, (uint8_t *)pool, layer, p, b, 0), (size_t)g->Rp);"),
    "scatter_back_object_layer_term_dropped": (
        "const uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride",
        "const uint8_t *obj = q->objects + 0 * q->obj_layer_stride"),
    "scatter_back_object_plane_term_dropped": (
        "const uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride\n"
        "                                   + (int64_t)p * q->obj_plane_stride",
        "const uint8_t *obj = q->objects + (int64_t)layer * q->obj_layer_stride\n"
        "                                   + 0 * q->obj_plane_stride"),
    "scatter_back_writes_layer_zero": (
        "memcpy(pool_slot(g, pool, layer, p, b, 0), obj, (size_t)obj_bytes);",
        "memcpy(pool_slot(g, pool, 0, p, b, 0), obj, (size_t)obj_bytes);"),
    "scatter_back_ignores_request_table_offset": (
        "                int64_t b = tables[tab0 + j];\n"
        "                if (b < 0 || b >= g->n_pool) { note(&status, OR_ERANGE); continue; }\n"
        "                const uint8_t",
        "                int64_t b = tables[j];\n"
        "                if (b < 0 || b >= g->n_pool) { note(&status, OR_ERANGE); continue; }\n"
        "                const uint8_t"),
}

PIN_CALLS = [
    (pins.test_block_and_object_counts_match_tutti, dict(row=pins.golden_counts()[1], hit_frac=0.75)),
    (pins.test_object_bytes_equal_tutti_eq1, {}),
    (pins.test_merge_scatter_places_hit_then_miss_tokens, dict(source="permuted", miss_order="layer")),
    (pins.test_slice_and_concatenate_keep_token_layer_plane_order, dict(source="permuted")),
    (pins.test_gather_objects_hold_blocks_in_table_order, {}),
    (pins.test_block_major_objects_form_one_file_of_2L_objects_per_block, {}),
    (pins.test_identity_table_pool_is_a_reshape_of_complete_layer, {}),
    (pins.test_scatter_back_after_gather_restores_the_pool, {}),
    (pins.test_oracle_matches_brute_force, dict(case=1)),
    (pins.test_plan_prefix_sums_and_work_list, {}),
    (pins.test_plan_flags_planted_errors, {}),
]


def _build_mutant(tmp_path, name):
    src = oracle.SRC.read_text()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation {name} does not apply"
    mutated = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c99", "-shared", "-fPIC", str(c), "-o", str(so)],
                   check=True)
    return oracle.load_library(so)


def test_unmutated_oracle_passes_every_pin_call():
    lib = oracle.load_library()
    for fn, kw in PIN_CALLS:
        fn(**kw, lib=lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    caught = []
    for fn, kw in PIN_CALLS:
        try:
            fn(**kw, lib=lib)
        except AssertionError:
            caught.append(fn.__name__)
    # the brute-force restatement is a second implementation, not a pin to the pages:
    # some pin besides it has to see the mistake
    assert set(caught) - {"test_oracle_matches_brute_force"}, \
        f"no pin other than the brute force caught mutation {name} ({caught})"
