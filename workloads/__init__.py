"""Seeded synthetic inputs for the layer-wise paged KV block reshuffle.

This module builds INPUTS only: the shapes, hit/miss token counts, block tables and
KV payload of each workload, and where each request's buffers sit in a few packed
byte buffers.  It holds none of the reshuffle itself (no slicing, merging, scattering
or gathering); both the CUDA path and the CPU oracle consume what it builds.

Workloads (named by what they are):

* ``tiny``               -- L=2, H_kv=2, d=64, B=16, one request 96 hit + 32 miss tokens,
                            a 32-block pool, block table = seeded random permutation.
* ``llama3_8b_agentic``  -- L=32, H_kv=8, d=128, B=16, one request 30720 hit + 512 miss,
                            full-block source [T_hit, 32, 2, 8, 128], 4096-block pool with
                            a shuffled block table.
* ``qwen3_32b_long``     -- L=64, H_kv=8, d=128, B=64, T=128000 at 75 % hit, values
                            uniform in [-2, 2], source full blocks and pool both permuted.
* ``latent_batch``       -- latent KV: C_KV=576 (one plane), L=61, B=64, 16 requests with
                            T_hit ~ U[16384, 49152], T_miss ~ U[128, 2048], one shared pool.
* ``many_small``         -- L=32, H_kv=8, d=128, B=16, 256 requests, T_hit lognormal
                            (median 2048, sigma 0.5, clipped to [256, 8192]),
                            T_miss ~ U[16, 256], tables from a fragmented free list.

Geometry symbols follow the pages: L layers, B tokens per paged block, P planes
(2 = K and V for head-split KV, 1 = a latent vector), Rp bytes per token per plane
(H_kv*d*2 for bf16, C_KV*2 for latent), R = P*Rp bytes per token row of one layer.

Readings taken where the workload text is silent (each listed in the design notes):
the lognormal sigma is 0.5; the pool for the batched workloads holds
ceil(1.25 * sum of blocks) blocks; "fragmented free list" = the pool ids cut into runs
of U[1, 8] consecutive ids, the runs shuffled, then handed out in order; a "permuted
source" stores the hit prefix as whole full blocks [B, L, P, Rp] at shuffled positions.
Seeds are 20261200 + k for the k-th workload.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

BF16_BYTES = 2

# Fill byte for buffers the reshuffle writes (pool, objects, outputs): any byte the
# reshuffle does not write keeps this value, which makes partial blocks visible.
SENTINEL = 0xA5


@dataclass(frozen=True)
class Spec:
    """One workload: geometry, per-request token counts, table and value recipes."""
    name: str
    L: int                      # layers
    P: int                      # planes per token (2 = K,V ; 1 = latent)
    B: int                      # tokens per paged block
    Rp: int                     # bytes per token per plane
    t_hit: tuple                # per request
    t_miss: tuple               # per request
    n_pool: int                 # physical blocks in the paged pool
    values: str = "normal"      # "normal" | "uniform2" | "bytes"
    table: str = "perm"         # "perm" | "shared_perm" | "fragmented" | "identity"
    source: str = "contiguous"  # "contiguous" ([T_hit, L, P, Rp]) | "permuted" (blocks)
    miss_order: str = "layer"   # "layer" ([L, T_miss, P, Rp]) | "token" ([T_miss, L, P, Rp])
    seed: int = 0
    objects: str = "layer"      # "layer" ([L][P][nblk][B][Rp]) | "block" ([nblk][L][P][B][Rp])
    # One rank's part of a batch split across GPUs (layer_wise_paged_gb300.shard): its
    # block tables, renumbered into its own pool, and its full-block tables replace the
    # recipes above; `part` names the part ("" for a whole batch).
    given_tables: object = field(default=None, compare=False, repr=False)
    given_src_tables: object = field(default=None, compare=False, repr=False)
    part: str = ""

    @property
    def R(self) -> int:
        return self.P * self.Rp

    @property
    def n_req(self) -> int:
        return len(self.t_hit)

    def t_all(self) -> np.ndarray:
        return np.asarray(self.t_hit, np.int64) + np.asarray(self.t_miss, np.int64)

    def nblk(self) -> np.ndarray:
        """Paged blocks each request occupies, ceil(T_all / B)."""
        return -(-self.t_all() // self.B)

    def nsrc(self) -> np.ndarray:
        """Full blocks holding each request's hit prefix, ceil(T_hit / B)."""
        return -(-np.asarray(self.t_hit, np.int64) // self.B)


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def get_spec(name: str) -> Spec:
    """The five named workloads, with their counts drawn from the workload's seed."""
    if name == "tiny":
        return Spec("tiny", L=2, P=2, B=16, Rp=2 * 64 * BF16_BYTES, t_hit=(96,), t_miss=(32,),
                    n_pool=32, values="normal", table="perm", seed=20261201)
    if name == "llama3_8b_agentic":
        return Spec(name, L=32, P=2, B=16, Rp=8 * 128 * BF16_BYTES, t_hit=(30720,), t_miss=(512,),
                    n_pool=4096, values="normal", table="perm", seed=20261202)
    if name == "qwen3_32b_long":
        return Spec(name, L=64, P=2, B=64, Rp=8 * 128 * BF16_BYTES, t_hit=(96000,), t_miss=(32000,),
                    n_pool=2048, values="uniform2", table="perm", source="permuted",
                    seed=20261203)
    if name == "latent_batch":
        seed = 20261204
        g = _rng(seed)
        t_hit = tuple(int(x) for x in g.integers(16384, 49152, size=16, endpoint=True))
        t_miss = tuple(int(x) for x in g.integers(128, 2048, size=16, endpoint=True))
        s = Spec(name, L=61, P=1, B=64, Rp=576 * BF16_BYTES, t_hit=t_hit, t_miss=t_miss,
                 n_pool=1, values="normal", table="shared_perm", seed=seed)
        return replace(s, n_pool=int(math.ceil(1.25 * int(s.nblk().sum()))))
    if name == "many_small":
        seed = 20261205
        g = _rng(seed)
        raw = g.lognormal(mean=math.log(2048.0), sigma=0.5, size=256)
        t_hit = tuple(int(x) for x in np.clip(np.rint(raw), 256, 8192))
        t_miss = tuple(int(x) for x in g.integers(16, 256, size=256, endpoint=True))
        s = Spec(name, L=32, P=2, B=16, Rp=8 * 128 * BF16_BYTES, t_hit=t_hit, t_miss=t_miss,
                 n_pool=1, values="normal", table="fragmented", seed=seed)
        return replace(s, n_pool=int(math.ceil(1.25 * int(s.nblk().sum()))))
    raise KeyError(name)


NAMES = ("tiny", "llama3_8b_agentic", "qwen3_32b_long", "latent_batch", "many_small")


def custom_spec(name="custom", *, L, P, B, Rp, t_hit, t_miss, n_pool=None, values="bytes",
                table="perm", source="contiguous", miss_order="layer", seed=1,
                objects="layer") -> Spec:
    """A small ad-hoc workload for tests (pool defaults to 1.5x the blocks needed)."""
    s = Spec(name, L=L, P=P, B=B, Rp=Rp, t_hit=tuple(int(x) for x in t_hit),
             t_miss=tuple(int(x) for x in t_miss), n_pool=1, values=values, table=table,
             source=source, miss_order=miss_order, seed=seed, objects=objects)
    if n_pool is None:
        n_pool = max(1, int(math.ceil(1.5 * max(1, int(s.nblk().sum())))))
    return replace(s, n_pool=int(n_pool))


def part_spec(spec: Spec, part):
    """The workload of one rank's part of `spec` (a layer_wise_paged_gb300.shard.Part):
    its requests and layers, a pool of the blocks it uses, its renumbered tables; None
    for an idle rank.  The payload is drawn from the workload's seed as for any spec."""
    if part.kind == "idle":
        return None
    idx = list(part.requests)
    l0, l1 = part.layers
    return replace(spec, L=l1 - l0, t_hit=tuple(spec.t_hit[i] for i in idx),
                   t_miss=tuple(spec.t_miss[i] for i in idx),
                   n_pool=max(1, int(len(part.pool_ids))), given_tables=part.tables,
                   given_src_tables=part.src_tables,
                   part=f"rank {part.rank} of {part.world}: {part.kind} "
                        + (f"{idx[0]}..{idx[-1]}" if part.kind == "requests" else f"layers {l0}..{l1 - 1}"))


def block_tables(spec: Spec) -> np.ndarray:
    """Per-request block tables, packed back to back in request order (int32).

    Request r's table is the next nblk(r) entries.  Every recipe is injective into
    [0, n_pool) provided the pool holds at least sum(nblk) blocks.
    """
    nblk = spec.nblk()
    total = int(nblk.sum())
    if spec.given_tables is not None:
        return np.ascontiguousarray(spec.given_tables, dtype=np.int32)
    g = _rng(spec.seed + 1)
    if total > spec.n_pool:
        raise ValueError(f"{spec.name}: {total} blocks needed, pool holds {spec.n_pool}")
    if spec.table == "identity":
        flat = np.arange(total, dtype=np.int64)
    elif spec.table in ("perm", "shared_perm"):
        flat = g.permutation(spec.n_pool)[:total]
    elif spec.table == "fragmented":
        runs, start = [], 0
        while start < spec.n_pool:
            n = int(g.integers(1, 8, endpoint=True))
            runs.append(np.arange(start, min(start + n, spec.n_pool)))
            start += n
        order = g.permutation(len(runs))
        flat = np.concatenate([runs[i] for i in order])[:total]
    else:
        raise KeyError(spec.table)
    return np.ascontiguousarray(flat, dtype=np.int32)


def source_tables(spec: Spec):
    """Per-request full-block tables for a permuted source (None for a contiguous one).

    Request r's hit prefix is stored as nsrc(r) full blocks of [B, L, P, Rp]; its table
    (the next nsrc(r) entries, packed in request order) maps logical full block j to
    the position where that block is stored in the request's source buffer.
    """
    if spec.source == "contiguous":
        return None
    if spec.given_src_tables is not None:
        return np.ascontiguousarray(spec.given_src_tables, dtype=np.int32)
    g = _rng(spec.seed + 2)
    parts = [g.permutation(int(n)) for n in spec.nsrc()]
    if not parts:
        return np.zeros(0, np.int32)
    return np.ascontiguousarray(np.concatenate(parts), dtype=np.int32)


@dataclass
class RequestLayout:
    """Byte offsets (into the packed buffers) and byte strides of one request."""
    t_hit: int
    t_miss: int
    hit_off: int
    hit_src_blocks: int
    hit_block_stride: int
    hit_token_stride: int
    hit_layer_stride: int
    src_table_off: int          # entry offset into the packed source tables, -1 = none
    miss_off: int
    miss_token_stride: int
    miss_layer_stride: int
    obj_off: int
    obj_layer_stride: int
    obj_plane_stride: int
    obj_block_stride: int


@dataclass
class Layout:
    spec: Spec
    requests: list = field(default_factory=list)
    hit_bytes: int = 0          # packed full-block buffer
    miss_bytes: int = 0         # packed miss buffer
    obj_bytes: int = 0          # packed objects buffer
    pool_bytes: int = 0
    hit_out_bytes: int = 0      # one layer of hit rows, all requests
    complete_bytes: int = 0     # one layer of complete rows, all requests


def layout(spec: Spec, *, objects_one_layer: bool = False) -> Layout:
    """Where each request's inputs and objects sit in the packed buffers.

    objects_one_layer=True gives every request an object region of one layer and
    object layer stride 0, so each layer's gather lands in the same place (used to
    bound memory on the largest workloads; checked layer by layer).
    """
    L, P, B, R = spec.L, spec.P, spec.B, spec.R
    out = Layout(spec)
    hit = miss = obj = 0
    nblk = spec.nblk()
    nsrc = spec.nsrc()
    src_tab = 0
    for r in range(spec.n_req):
        th, tm = int(spec.t_hit[r]), int(spec.t_miss[r])
        if spec.source == "contiguous":
            hb = th * L * R
            rl_src = dict(hit_src_blocks=int(nsrc[r]), hit_block_stride=B * L * R,
                          hit_token_stride=L * R, hit_layer_stride=R, src_table_off=-1)
        else:
            hb = int(nsrc[r]) * B * L * R
            rl_src = dict(hit_src_blocks=int(nsrc[r]), hit_block_stride=B * L * R,
                          hit_token_stride=L * R, hit_layer_stride=R, src_table_off=src_tab)
            src_tab += int(nsrc[r])
        if spec.miss_order == "layer":
            miss_strides = dict(miss_token_stride=R, miss_layer_stride=tm * R)
        else:
            miss_strides = dict(miss_token_stride=L * R, miss_layer_stride=R)
        nb, obj_sz = int(nblk[r]), B * spec.Rp
        per_layer_obj = P * nb * obj_sz
        ob = per_layer_obj if objects_one_layer else L * per_layer_obj
        if spec.objects == "layer":
            obj_strides = dict(obj_layer_stride=per_layer_obj, obj_plane_stride=nb * obj_sz,
                               obj_block_stride=obj_sz)
        elif spec.objects == "block":  # one file per block holding its 2L objects
            obj_strides = dict(obj_layer_stride=P * obj_sz, obj_plane_stride=obj_sz,
                               obj_block_stride=(1 if objects_one_layer else L) * P * obj_sz)
        else:
            raise KeyError(spec.objects)
        if objects_one_layer:
            obj_strides["obj_layer_stride"] = 0
        out.requests.append(RequestLayout(
            t_hit=th, t_miss=tm, hit_off=hit, **rl_src, miss_off=miss, **miss_strides,
            obj_off=obj, **obj_strides))
        hit += hb
        miss += L * tm * R
        obj += ob
    out.hit_bytes, out.miss_bytes, out.obj_bytes = hit, miss, obj
    out.pool_bytes = L * P * spec.n_pool * B * spec.Rp
    out.hit_out_bytes = int(sum(spec.t_hit)) * R
    out.complete_bytes = int(spec.t_all().sum()) * R
    return out


HOST_BLOCK = 256 << 20  # CPU payloads repeat a seeded block of this many bytes


def fill_payload(buf, kind: str, seed: int) -> None:
    """Fill a torch uint8 buffer (CPU or CUDA) with seeded KV payload, in place.

    "normal" = bf16 N(0, 1), "uniform2" = bf16 uniform in [-2, 2], "bytes" = uniform
    random bytes (every bit pattern, NaNs, -0.0 and subnormals included).  On the GPU
    every byte is drawn; on the CPU a buffer longer than HOST_BLOCK repeats its first
    HOST_BLOCK bytes (the reshuffle copies bytes, so only the value distribution
    matters, and drawing tens of GB on the host would take minutes).
    """
    import torch
    n = buf.numel()
    if n == 0:
        return
    g = torch.Generator(device=buf.device)
    g.manual_seed(seed)
    chunk = 1 << 30 if buf.device.type == "cuda" else HOST_BLOCK
    for s in range(0, n, chunk):
        part = buf[s:min(n, s + chunk)]
        if buf.device.type != "cuda" and s > 0:
            part.copy_(buf[:part.numel()])
        elif kind == "bytes" or part.numel() % 2:
            part.copy_(torch.randint(0, 256, (part.numel(),), generator=g, device=buf.device,
                                     dtype=torch.int32).to(torch.uint8))
        elif kind == "normal":
            part.view(torch.bfloat16).normal_(0.0, 1.0, generator=g)
        elif kind == "uniform2":
            part.view(torch.bfloat16).uniform_(-2.0, 2.0, generator=g)
        else:
            raise KeyError(kind)


def allocate(spec: Spec, device, *, objects_one_layer: bool = False, fill: bool = True):
    """Allocate and fill every buffer of a workload on `device` (torch uint8 tensors).

    Returns a dict with the layout, the packed hit/miss/object buffers, the pool
    (sentinel-filled), the block tables and the source tables (int32 tensors).
    """
    import torch
    lay = layout(spec, objects_one_layer=objects_one_layer)
    dev = torch.device(device)

    def u8(nbytes, sentinel):
        t = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=dev)
        if sentinel:
            t.fill_(SENTINEL)
        return t

    bufs = dict(layout=lay)
    bufs["hit"] = u8(lay.hit_bytes, False)
    bufs["miss"] = u8(lay.miss_bytes, False)
    if fill:
        fill_payload(bufs["hit"], spec.values, spec.seed * 7 + 1)
        fill_payload(bufs["miss"], spec.values, spec.seed * 7 + 2)
    bufs["pool"] = u8(lay.pool_bytes, True)
    bufs["objects"] = u8(lay.obj_bytes, True)
    tables = block_tables(spec)
    bufs["tables"] = torch.from_numpy(tables if tables.size else np.zeros(1, np.int32)).to(dev)
    st = source_tables(spec)
    bufs["src_tables"] = None if st is None else torch.from_numpy(
        st if st.size else np.zeros(1, np.int32)).to(dev)
    return bufs


def footprint_bytes(spec: Spec, *, objects_one_layer: bool = False) -> int:
    """Device bytes `allocate` needs (inputs, pool, objects, tables)."""
    lay = layout(spec, objects_one_layer=objects_one_layer)
    return lay.hit_bytes + lay.miss_bytes + lay.pool_bytes + lay.obj_bytes + 8 * int(spec.nblk().sum())
