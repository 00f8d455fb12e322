"""CPU oracle of the layer-wise paged KV block reshuffle (test infrastructure).

TEST INFRASTRUCTURE ONLY: only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package.  The product path never does,
and this package never imports the product package.

The arithmetic lives in ``kvl_oracle.c``: plain nested loops over requests, tokens,
planes and blocks, in the order the pages give the steps (slice_layer,
concatenate_tokens, scatter into the paged pool, gather into per-layer K/V objects,
scatter back).  This module only compiles that file with gcc, loads it with ctypes
and marshals numpy arrays into it.

Pins: every function here is checked against what the pages and the mathematics fix
(block and object counts of Tutti eqs. (3)(4)(14)(15), the KV size of eq. (1),
hit-before-miss and token/layer/head order by tagged payloads, reshape special cases,
round trips, and a pure-Python brute force on tiny inputs) in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "kvl_oracle.c"
BUILD_DIR = HERE / "_build"
LIB = BUILD_DIR / "libkvl_oracle.so"

OK, EINVAL, ERANGE, EDUP = 0, 1, 3, 4


def build(force: bool = False) -> Path:
    """Compile the oracle into a shared library with gcc (plain C99, -O2)."""
    BUILD_DIR.mkdir(exist_ok=True)
    if force or not LIB.exists() or LIB.stat().st_mtime < SRC.stat().st_mtime:
        tmp = LIB.with_suffix(f".so.{os.getpid()}")
        subprocess.run(["gcc", "-O2", "-std=c99", "-Wall", "-shared", "-fPIC",
                        str(SRC), "-o", str(tmp)], check=True)
        os.replace(tmp, LIB)
    return LIB


class _Geom(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("P", ctypes.c_int32), ("B", ctypes.c_int32),
                ("Rp", ctypes.c_int32), ("n_pool", ctypes.c_int64)]


class _Req(ctypes.Structure):
    _fields_ = [("hit_src", ctypes.c_void_p), ("hit_src_table", ctypes.c_void_p),
                ("hit_src_blocks", ctypes.c_int64), ("hit_block_stride", ctypes.c_int64),
                ("hit_token_stride", ctypes.c_int64), ("hit_layer_stride", ctypes.c_int64),
                ("miss_src", ctypes.c_void_p), ("miss_token_stride", ctypes.c_int64),
                ("miss_layer_stride", ctypes.c_int64), ("objects", ctypes.c_void_p),
                ("obj_layer_stride", ctypes.c_int64), ("obj_plane_stride", ctypes.c_int64),
                ("obj_block_stride", ctypes.c_int64), ("t_hit", ctypes.c_int32),
                ("t_miss", ctypes.c_int32)]


_lib = None


def load_library(path=None):
    """Load the oracle library (the default build, or another build of the same source
    at `path`, which the mutation tests use to check that the pins catch mistakes)."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(str(build() if path is None else path))
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.oracle_plan.argtypes = [i32, p, i32, p, i64, i32, i64, p, p, p, p, p, p, p]
    lib.oracle_slice_layer.argtypes = [p, i32, p, i32, p]
    lib.oracle_concatenate_tokens.argtypes = [p, i32, p, i32, p, p]
    lib.oracle_scatter_paged.argtypes = [p, i32, p, p, i32, p, p]
    lib.oracle_merge_scatter.argtypes = [p, i32, p, p, i32, p, p]
    lib.oracle_gather_objects.argtypes = [p, i32, p, p, i32, p]
    lib.oracle_scatter_back.argtypes = [p, i32, p, p, i32, p]
    for f in (lib.oracle_plan, lib.oracle_slice_layer, lib.oracle_concatenate_tokens,
              lib.oracle_scatter_paged, lib.oracle_merge_scatter,
              lib.oracle_gather_objects, lib.oracle_scatter_back):
        f.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(a: np.ndarray | None, off: int = 0):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data + off


class Batch:
    """One batch of requests over host (numpy) buffers.

    geom: object with L, P, B, Rp, n_pool.  requests: sequence of objects with the
    byte-layout attributes t_hit, t_miss, hit_off, hit_src_blocks, hit_block_stride,
    hit_token_stride, hit_layer_stride, src_table_off, miss_off, miss_token_stride,
    miss_layer_stride, obj_off, obj_layer_stride, obj_plane_stride, obj_block_stride.
    hit, miss, objects: uint8 numpy
    buffers the offsets index; src_tables: packed int32 full-block tables or None;
    tables: packed int32 pool block tables (request order).
    """

    def __init__(self, geom, requests, hit, miss, objects, tables, src_tables=None, lib=None):
        self._lib = lib if lib is not None else load_library()
        self.g = _Geom(int(geom.L), int(geom.P), int(geom.B), int(geom.Rp), int(geom.n_pool))
        self.L, self.P, self.B, self.Rp, self.n_pool = (int(geom.L), int(geom.P), int(geom.B),
                                                         int(geom.Rp), int(geom.n_pool))
        self.R = self.P * self.Rp
        self.hit, self.miss, self.objects = hit, miss, objects
        self.tables = np.ascontiguousarray(tables, dtype=np.int32)
        self.src_tables = None if src_tables is None else np.ascontiguousarray(src_tables, np.int32)
        self.n_req = len(requests)
        self.reqs = (_Req * max(1, self.n_req))()
        self.t_hit = np.array([int(q.t_hit) for q in requests], np.int64)
        self.t_miss = np.array([int(q.t_miss) for q in requests], np.int64)
        for r, q in enumerate(requests):
            x = self.reqs[r]
            x.hit_src = _ptr(hit, int(q.hit_off)) if hit is not None and hit.size else None
            if q.src_table_off is not None and q.src_table_off >= 0:
                x.hit_src_table = _ptr(self.src_tables, 4 * int(q.src_table_off))
            else:
                x.hit_src_table = None
            x.hit_src_blocks = int(q.hit_src_blocks)
            x.hit_block_stride = int(q.hit_block_stride)
            x.hit_token_stride = int(q.hit_token_stride)
            x.hit_layer_stride = int(q.hit_layer_stride)
            x.miss_src = _ptr(miss, int(q.miss_off)) if miss is not None and miss.size else None
            x.miss_token_stride = int(q.miss_token_stride)
            x.miss_layer_stride = int(q.miss_layer_stride)
            x.objects = _ptr(objects, int(q.obj_off)) if objects is not None and objects.size else None
            x.obj_layer_stride = int(q.obj_layer_stride)
            x.obj_plane_stride = int(q.obj_plane_stride)
            x.obj_block_stride = int(q.obj_block_stride)
            x.t_hit = int(q.t_hit)
            x.t_miss = int(q.t_miss)

    # -- counts ------------------------------------------------------------
    def total_hit(self) -> int:
        return int(np.clip(self.t_hit, 0, None).sum())

    def total_tokens(self) -> int:
        return int((np.clip(self.t_hit, 0, None) + np.clip(self.t_miss, 0, None)).sum())

    # -- the steps ---------------------------------------------------------
    def plan(self, check_injective: bool = True, capacity: int | None = None) -> dict:
        """Prefix sums and work list.  Returns status, detail, n_items and the arrays."""
        lib = self._lib
        n = self.n_req
        cap = self.n_pool if capacity is None else int(capacity)
        tok = np.zeros(n + 1, np.int64)
        hit = np.zeros(n + 1, np.int64)
        blk = np.zeros(n + 1, np.int64)
        n_est = max(1, int(sum(-(-max(0, int(a) + int(b)) // self.B)
                               for a, b in zip(self.t_hit, self.t_miss))))
        item_req = np.zeros(n_est, np.int32)
        item_blk = np.zeros(n_est, np.int32)
        n_items = np.zeros(1, np.int64)
        detail = np.zeros(1, np.int64)
        st = lib.oracle_plan(n, ctypes.addressof(self.reqs), self.B, _ptr(self.tables),
                             self.n_pool, int(bool(check_injective)), cap, _ptr(tok), _ptr(hit),
                             _ptr(blk), _ptr(item_req), _ptr(item_blk), _ptr(n_items),
                             _ptr(detail))
        k = int(n_items[0])
        return dict(status=int(st), detail=int(detail[0]), n_items=k, tok_off=tok,
                    hit_off=hit, blk_off=blk, item_req=item_req[:k], item_blk=item_blk[:k])

    def slice_layer(self, layer: int):
        lib = self._lib
        out = np.zeros(max(1, self.total_hit() * self.R), np.uint8)
        st = lib.oracle_slice_layer(ctypes.addressof(self.g), self.n_req,
                                    ctypes.addressof(self.reqs), int(layer), _ptr(out))
        return int(st), out[: self.total_hit() * self.R]

    def concatenate_tokens(self, layer: int, hit_layer: np.ndarray):
        lib = self._lib
        out = np.zeros(max(1, self.total_tokens() * self.R), np.uint8)
        hl = np.ascontiguousarray(hit_layer if hit_layer.size else np.zeros(1, np.uint8))
        st = lib.oracle_concatenate_tokens(ctypes.addressof(self.g), self.n_req,
                                           ctypes.addressof(self.reqs), int(layer), _ptr(hl),
                                           _ptr(out))
        return int(st), out[: self.total_tokens() * self.R]

    def scatter_paged(self, layer: int, complete_layer: np.ndarray, pool: np.ndarray) -> int:
        lib = self._lib
        cl = np.ascontiguousarray(complete_layer if complete_layer.size else np.zeros(1, np.uint8))
        return int(lib.oracle_scatter_paged(ctypes.addressof(self.g), self.n_req,
                                            ctypes.addressof(self.reqs), _ptr(self.tables),
                                            int(layer), _ptr(cl), _ptr(pool)))

    def merge_scatter(self, layer: int, pool: np.ndarray, want_complete: bool = False):
        """slice_layer, concatenate_tokens and the paged scatter of one layer."""
        lib = self._lib
        comp = np.zeros(max(1, self.total_tokens() * self.R), np.uint8) if want_complete else None
        st = lib.oracle_merge_scatter(ctypes.addressof(self.g), self.n_req,
                                      ctypes.addressof(self.reqs), _ptr(self.tables), int(layer),
                                      _ptr(pool), _ptr(comp))
        return int(st), (None if comp is None else comp[: self.total_tokens() * self.R])

    def gather_objects(self, layer: int, pool: np.ndarray) -> int:
        lib = self._lib
        return int(lib.oracle_gather_objects(ctypes.addressof(self.g), self.n_req,
                                             ctypes.addressof(self.reqs), _ptr(self.tables),
                                             int(layer), _ptr(pool)))

    def scatter_back(self, layer: int, pool: np.ndarray) -> int:
        lib = self._lib
        return int(lib.oracle_scatter_back(ctypes.addressof(self.g), self.n_req,
                                           ctypes.addressof(self.reqs), _ptr(self.tables),
                                           int(layer), _ptr(pool)))
