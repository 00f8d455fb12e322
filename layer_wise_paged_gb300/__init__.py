"""Python binding of libkvl.so: the layer-wise paged KV block reshuffle on one GB300.

Argument marshalling only.  Every step of the reshuffle (plan, slice, merge-scatter,
gather, scatter-back) runs in the library's CUDA kernels; this module turns Python
integers (device addresses, stream handles) and small host structs into the C ABI
declared in ``include/kvl.h``.  There is no CPU fallback: if the library is missing
the first call raises.

Pointers are plain integers (for a torch tensor, ``t.data_ptr()``); streams are
integers too (``torch.cuda.current_stream().cuda_stream``) or None for the legacy
default stream.
"""
from __future__ import annotations

import ctypes

import numpy as np

from .build import LIB, build

KVL_OK, KVL_EINVAL, KVL_EALIGN, KVL_ERANGE, KVL_EDUP, KVL_ECUDA, KVL_ETIMEOUT = range(7)
KVL_GATHER, KVL_SCATTER_BACK = 0, 1
STATUS_NAMES = {0: "KVL_OK", 1: "KVL_EINVAL", 2: "KVL_EALIGN", 3: "KVL_ERANGE", 4: "KVL_EDUP",
                5: "KVL_ECUDA", 6: "KVL_ETIMEOUT"}


class KvlError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = int(code)
        super().__init__(f"{what}: {STATUS_NAMES.get(self.code, self.code)} "
                         f"({kvl_status_string(self.code)})")


class kvl_launch(ctypes.Structure):
    _fields_ = [("max_ctas", ctypes.c_int32), ("flags", ctypes.c_int32)]


KVL_LAUNCH_HOST_SRC, KVL_LAUNCH_HOST_DST, KVL_LAUNCH_OVERLAP_PREVIOUS, KVL_LAUNCH_SHARE_SMS = 1, 2, 4, 8
KVL_LAUNCH_PLAN_READY = 16


class kvl_geom(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_planes", ctypes.c_int32),
                ("block_tokens", ctypes.c_int32), ("plane_row_bytes", ctypes.c_int32),
                ("pool_blocks", ctypes.c_int64)]


# struct kvl_request, 112 bytes, field for field
REQUEST_DTYPE = np.dtype([
    ("hit_src", np.uint64), ("hit_src_table", np.uint64), ("hit_src_blocks", np.int64),
    ("hit_block_stride", np.int64), ("hit_token_stride", np.int64),
    ("hit_layer_stride", np.int64), ("miss_src", np.uint64), ("miss_token_stride", np.int64),
    ("miss_layer_stride", np.int64), ("objects", np.uint64), ("obj_layer_stride", np.int64),
    ("obj_plane_stride", np.int64), ("obj_block_stride", np.int64),
    ("t_hit", np.int32), ("t_miss", np.int32)])
assert REQUEST_DTYPE.itemsize == 112

_lib = None


def lib():
    """The loaded libkvl.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not LIB.exists():
            raise RuntimeError(f"libkvl.so is not built ({LIB}); run "
                               "layer_wise_paged_gb300.build.build() first")
        L = ctypes.CDLL(str(LIB))
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        gp = ctypes.POINTER(kvl_geom)
        L.kvl_plan_bytes.argtypes, L.kvl_plan_bytes.restype = [gp, i32], sz
        L.kvl_plan_layout.argtypes, L.kvl_plan_layout.restype = [gp, i32, ctypes.POINTER(sz)], None
        L.kvl_batch_plan.argtypes = [gp, i32, vp, vp, i32, vp, sz, vp]
        L.kvl_batch_plan_static_scratch.argtypes = [gp, i32, vp, vp, i32, vp, sz, vp]
        lp = ctypes.POINTER(kvl_launch)
        L.kvl_slice_layer.argtypes = [gp, vp, sz, vp, i32, i32, vp, lp, vp]
        L.kvl_merge_scatter_paged.argtypes = [gp, vp, sz, vp, vp, i32, i32, vp, vp, lp, vp]
        L.kvl_gather_layer_objects.argtypes = [gp, vp, sz, vp, vp, i32, i32, vp, i32, lp, vp]
        L.kvl_read_status.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i64), vp]
        L.kvl_diag_wait_timeout.argtypes, L.kvl_diag_wait_timeout.restype = [i32, vp, vp], i32
        L.kvl_status_string.argtypes, L.kvl_status_string.restype = [i32], ctypes.c_char_p
        L.kvl_launches_per_call.argtypes, L.kvl_launches_per_call.restype = [i32], i32
        for f in (L.kvl_batch_plan, L.kvl_batch_plan_static_scratch, L.kvl_slice_layer, L.kvl_merge_scatter_paged,
                  L.kvl_gather_layer_objects, L.kvl_read_status):
            f.restype = i32
        _lib = L
    return _lib


def geom(L, P, B, Rp, N) -> kvl_geom:
    return kvl_geom(int(L), int(P), int(B), int(Rp), int(N))


def _g(g):
    if isinstance(g, kvl_geom):
        return ctypes.byref(g)
    return ctypes.byref(geom(*g))


def _p(x):
    return None if x is None or x == 0 else ctypes.c_void_p(int(x))


def _launch(max_ctas, flags=0):
    """Launch options: None (whole GPU, device buffers), a CTA cap, or a kvl_launch."""
    if isinstance(max_ctas, kvl_launch):
        return ctypes.byref(max_ctas)
    if max_ctas is None and not flags:
        return None
    return ctypes.byref(kvl_launch(int(max_ctas or 0), int(flags)))


def kvl_plan_bytes(g, n_req: int) -> int:
    return int(lib().kvl_plan_bytes(_g(g), int(n_req)))


def kvl_plan_layout(g, n_req: int) -> list:
    off = (ctypes.c_size_t * 11)()
    lib().kvl_plan_layout(_g(g), int(n_req), off)
    return [int(x) for x in off]


def kvl_batch_plan(g, n_req, d_reqs, d_block_tables, check_injective, d_plan, plan_bytes,
                   stream=None) -> int:
    return int(lib().kvl_batch_plan(_g(g), int(n_req), _p(d_reqs), _p(d_block_tables),
                                    int(bool(check_injective)), _p(d_plan), int(plan_bytes),
                                    _p(stream)))


def kvl_batch_plan_static_scratch(g, n_req, d_reqs, d_block_tables, check_injective, d_plan,
                                  plan_bytes, stream=None) -> int:
    """kvl_batch_plan for callers that cannot allocate device memory: its scratch is a
    fixed array inside the library (pool_blocks <= KVL_STATIC_SCRATCH_POOL_BLOCKS)."""
    return int(lib().kvl_batch_plan_static_scratch(_g(g), int(n_req), _p(d_reqs),
                                                   _p(d_block_tables), int(bool(check_injective)),
                                                   _p(d_plan), int(plan_bytes), _p(stream)))


KVL_STATIC_SCRATCH_POOL_BLOCKS = 1 << 22


def kvl_slice_layer(g, d_plan, plan_bytes, d_reqs, layer, layer_count, d_hit_out,
                    max_ctas=None, stream=None) -> int:
    return int(lib().kvl_slice_layer(_g(g), _p(d_plan), int(plan_bytes), _p(d_reqs), int(layer),
                                     int(layer_count), _p(d_hit_out), _launch(max_ctas),
                                     _p(stream)))


def kvl_merge_scatter_paged(g, d_plan, plan_bytes, d_reqs, d_block_tables, layer, layer_count,
                            d_pool, d_complete_out=None, max_ctas=None, stream=None) -> int:
    return int(lib().kvl_merge_scatter_paged(_g(g), _p(d_plan), int(plan_bytes), _p(d_reqs),
                                             _p(d_block_tables), int(layer), int(layer_count),
                                             _p(d_pool), _p(d_complete_out), _launch(max_ctas),
                                             _p(stream)))


def kvl_gather_layer_objects(g, d_plan, plan_bytes, d_reqs, d_block_tables, layer, layer_count,
                             d_pool, direction, max_ctas=None, stream=None) -> int:
    return int(lib().kvl_gather_layer_objects(_g(g), _p(d_plan), int(plan_bytes), _p(d_reqs),
                                              _p(d_block_tables), int(layer), int(layer_count),
                                              _p(d_pool), int(direction), _launch(max_ctas),
                                              _p(stream)))


def kvl_read_status(d_plan, stream=None):
    """(code, detail) of a plan; synchronises the stream.  Raises if the copy fails."""
    code, detail = ctypes.c_int32(-1), ctypes.c_int64(0)
    st = lib().kvl_read_status(_p(d_plan), ctypes.byref(code), ctypes.byref(detail), _p(stream))
    if st != KVL_OK:
        raise KvlError(st, "kvl_read_status")
    return int(code.value), int(detail.value)


def kvl_diag_wait_timeout(limit_us, d_status, stream=None) -> int:
    """Make the copy kernels' bounded wait run out (see include/kvl.h)."""
    return int(lib().kvl_diag_wait_timeout(int(limit_us), _p(d_status), _p(stream)))


def kvl_status_string(code: int) -> str:
    return lib().kvl_status_string(int(code)).decode()


def kvl_launches_per_call(which: int) -> int:
    return int(lib().kvl_launches_per_call(int(which)))


def check(code: int, what: str = "kvl") -> None:
    """Raise KvlError for a non-OK status."""
    if code != KVL_OK:
        raise KvlError(code, what)


def pack_requests(requests, *, hit_base=0, miss_base=0, obj_base=0, src_table_base=0):
    """struct kvl_request array (host numpy) for requests given as byte layouts.

    Each request object carries t_hit, t_miss, hit_off, hit_src_blocks, the hit
    strides, src_table_off (-1 = none), miss_off, the miss strides, obj_off and the
    object layer, plane and block strides; *_base are the device addresses the offsets are relative to
    (src_table_off counts int32 entries).  A zero base leaves that pointer NULL.
    """
    out = np.zeros(max(1, len(requests)), REQUEST_DTYPE)
    for r, q in enumerate(requests):
        x = out[r]
        x["hit_src"] = hit_base + q.hit_off if hit_base and q.t_hit > 0 else 0
        x["hit_src_table"] = (src_table_base + 4 * q.src_table_off
                              if src_table_base and q.src_table_off >= 0 else 0)
        x["hit_src_blocks"] = q.hit_src_blocks
        x["hit_block_stride"] = q.hit_block_stride
        x["hit_token_stride"] = q.hit_token_stride
        x["hit_layer_stride"] = q.hit_layer_stride
        x["miss_src"] = miss_base + q.miss_off if miss_base and q.t_miss > 0 else 0
        x["miss_token_stride"] = q.miss_token_stride
        x["miss_layer_stride"] = q.miss_layer_stride
        x["objects"] = obj_base + q.obj_off if obj_base else 0
        x["obj_layer_stride"] = q.obj_layer_stride
        x["obj_plane_stride"] = q.obj_plane_stride
        x["obj_block_stride"] = q.obj_block_stride
        x["t_hit"] = q.t_hit
        x["t_miss"] = q.t_miss
    return out[:len(requests)] if requests else out[:0]


__all__ = ["build", "lib", "geom", "kvl_geom", "kvl_launch", "KVL_LAUNCH_HOST_SRC",
           "KVL_LAUNCH_HOST_DST", "REQUEST_DTYPE", "pack_requests", "check",
           "KvlError", "kvl_plan_bytes", "kvl_plan_layout", "kvl_batch_plan", "kvl_batch_plan_static_scratch",
           "kvl_slice_layer",
           "kvl_merge_scatter_paged", "kvl_gather_layer_objects", "kvl_read_status",
           "kvl_status_string", "kvl_launches_per_call"]
