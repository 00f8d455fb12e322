"""A batch of requests bound to device buffers: marshalling around the C ABI.

Holds the device copy of the ``kvl_request`` array, the block tables and the plan
buffer (torch tensors; PyTorch only provides device memory and streams), and
forwards each step to libkvl.so.  No step runs here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (KVL_GATHER, KVL_SCATTER_BACK, check, geom, kvl_batch_plan, kvl_launch,
               kvl_gather_layer_objects, kvl_merge_scatter_paged, kvl_plan_bytes,
               kvl_plan_layout, kvl_read_status, kvl_slice_layer, pack_requests)


def _ptr(t):
    return 0 if t is None else t.data_ptr()


class MappedHost:
    """Pinned host memory mapped into the device address space (cudaHostAlloc with
    cudaHostAllocMapped), for buffers a copy call reads or writes with the
    KVL_LAUNCH_HOST_SRC / KVL_LAUNCH_HOST_DST flags: `.np` is the host view (uint8),
    `data_ptr()` the device address."""

    _rt = None

    def __init__(self, nbytes):
        import ctypes
        if MappedHost._rt is None:
            torch.cuda.init()
            MappedHost._rt = ctypes.CDLL("libcudart.so.13")
        rt = MappedHost._rt
        self.nbytes = max(16, int(nbytes))
        self._h = ctypes.c_void_p()
        if rt.cudaHostAlloc(ctypes.byref(self._h), ctypes.c_size_t(self.nbytes),
                            ctypes.c_uint(2)) != 0:  # cudaHostAllocMapped
            raise MemoryError(f"cudaHostAlloc of {self.nbytes} bytes failed")
        d = ctypes.c_void_p()
        if rt.cudaHostGetDevicePointer(ctypes.byref(d), self._h, ctypes.c_uint(0)) != 0:
            raise RuntimeError("cudaHostGetDevicePointer failed")
        self._d = d.value
        buf = (ctypes.c_uint8 * self.nbytes).from_address(self._h.value)
        self.np = np.ctypeslib.as_array(buf)

    def data_ptr(self):
        return self._d

    def __del__(self):
        try:
            if self._h:
                MappedHost._rt.cudaFreeHost(self._h)
                self._h = None
        except Exception:
            pass


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Batch:
    """Requests of one batch over device buffers.

    g: (L, P, B, Rp, N).  requests: byte layouts (see ``pack_requests``).
    hit, miss, objects: torch uint8 device tensors the layouts' offsets index (or
    None).  tables: int32 device tensor of the packed block tables.  src_tables:
    int32 device tensor of packed full-block tables, or None.

    The copy calls take `layer_count` (layers per launch), `max_ctas` (at most that
    many SMs) and `flags`, the KVL_LAUNCH_* bits of include/kvl.h: host-memory
    sources or destinations, KVL_LAUNCH_OVERLAP_PREVIOUS (may run beside the launch
    before it, which must touch other bytes) and KVL_LAUNCH_SHARE_SMS.
    """

    def __init__(self, g, requests, hit, miss, objects, tables, src_tables=None):
        self.g = geom(*g)
        self.L, self.P, self.B, self.Rp, self.N = (int(x) for x in g)
        self.R = self.P * self.Rp
        self.requests = list(requests)
        self.n_req = len(self.requests)
        self.device = tables.device
        self.tables = tables
        self.src_tables = src_tables
        self.hit, self.miss, self.objects = hit, miss, objects
        host = pack_requests(self.requests, hit_base=_ptr(hit), miss_base=_ptr(miss),
                             obj_base=_ptr(objects), src_table_base=_ptr(src_tables))
        raw = np.ascontiguousarray(host).view(np.uint8).reshape(-1)
        if raw.size == 0:
            raw = np.zeros(112, np.uint8)
        self.d_reqs = torch.from_numpy(raw.copy()).to(self.device)
        self.plan_bytes = kvl_plan_bytes(self.g, self.n_req)
        self.d_plan = torch.zeros(self.plan_bytes, dtype=torch.uint8, device=self.device)
        self.layout = kvl_plan_layout(self.g, self.n_req)
        self.total_hit = int(sum(q.t_hit for q in self.requests))
        self.total_tokens = int(sum(q.t_hit + q.t_miss for q in self.requests))
        self.n_items = int(sum(-(-(q.t_hit + q.t_miss) // self.B) for q in self.requests))

    @staticmethod
    def _opts(max_ctas, flags):
        if not flags:
            return max_ctas
        return kvl_launch(int(max_ctas or 0), int(flags))

    # -- steps --------------------------------------------------------------
    def plan(self, check_injective=True, stream=None):
        check(kvl_batch_plan(self.g, self.n_req, _ptr(self.d_reqs), _ptr(self.tables),
                             check_injective, _ptr(self.d_plan), self.plan_bytes,
                             _stream(stream)), "kvl_batch_plan")

    def slice_layer(self, layer, hit_out, stream=None, layer_count=1, max_ctas=None, flags=0):
        check(kvl_slice_layer(self.g, _ptr(self.d_plan), self.plan_bytes, _ptr(self.d_reqs),
                              layer, layer_count, _ptr(hit_out), self._opts(max_ctas, flags),
                              _stream(stream)), "kvl_slice_layer")

    def merge_scatter(self, layer, pool, complete_out=None, stream=None, layer_count=1,
                      max_ctas=None, flags=0):
        check(kvl_merge_scatter_paged(self.g, _ptr(self.d_plan), self.plan_bytes,
                                      _ptr(self.d_reqs), _ptr(self.tables), layer, layer_count,
                                      _ptr(pool),
                                      _ptr(complete_out), self._opts(max_ctas, flags),
                                      _stream(stream)), "kvl_merge_scatter_paged")

    def gather(self, layer, pool, stream=None, layer_count=1, max_ctas=None, flags=0):
        check(kvl_gather_layer_objects(self.g, _ptr(self.d_plan), self.plan_bytes,
                                       _ptr(self.d_reqs), _ptr(self.tables), layer, layer_count,
                                       _ptr(pool),
                                       KVL_GATHER, self._opts(max_ctas, flags), _stream(stream)),
              "kvl_gather_layer_objects")

    def scatter_back(self, layer, pool, stream=None, layer_count=1, max_ctas=None, flags=0):
        check(kvl_gather_layer_objects(self.g, _ptr(self.d_plan), self.plan_bytes,
                                       _ptr(self.d_reqs), _ptr(self.tables), layer, layer_count,
                                       _ptr(pool),
                                       KVL_SCATTER_BACK, self._opts(max_ctas, flags),
                                       _stream(stream)), "kvl_gather_layer_objects")

    def status(self, stream=None):
        """(code, detail) of the plan after everything enqueued so far (synchronises)."""
        return kvl_read_status(_ptr(self.d_plan), _stream(stream))

    # -- plan contents (for tests) -----------------------------------------
    def plan_arrays(self):
        off, n = self.layout, self.n_req
        p = self.d_plan.cpu().numpy()
        hdr_i32 = p[:128].view(np.int32)
        hdr_i64 = p[:128].view(np.int64)
        n_items = int(hdr_i64[2])
        k = max(0, min(n_items, self.N))
        return dict(
            status=int(hdr_i32[0]), magic=int(hdr_i32[1]) & 0xffffffff, n_items=n_items,
            n_tokens=int(hdr_i64[3]), n_hit=int(hdr_i64[4]),
            tok_off=p[off[1]:off[1] + 8 * (n + 1)].view(np.int64).copy(),
            hit_off=p[off[2]:off[2] + 8 * (n + 1)].view(np.int64).copy(),
            blk_off=p[off[3]:off[3] + 8 * (n + 1)].view(np.int64).copy(),
            item_req=p[off[4]:off[4] + 4 * k].view(np.int32).copy(),
            item_blk=p[off[5]:off[5] + 4 * k].view(np.int32).copy())
