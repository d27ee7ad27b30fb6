"""Python face of the C ABI.  Functions keep the C names; they turn torch
tensors into pointers, sizes and the current CUDA stream and call the
library.  PyTorch is used only to own device memory and streams.
"""
from __future__ import annotations

import ctypes as C
import math
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _lib as L
from ._lib import check, lib

__all__ = [
    "dtype_code", "torch_dtype", "cb_rope_table_init", "cb_rope_reposition",
    "cb_kv_deviation_topk", "cb_kv_deviation_topk_noalloc", "cb_gather_rows",
    "cb_scatter_kv",
    "cb_sparse_query_attention", "cb_debug_expire_wait", "cb_debug_gemm_path", "Seg", "Req",
    "BlendModel", "ChunkStore", "HostChunkStore", "RollingWindow", "selection_stats",
    "loading_controller",
    "device_status",
]

device_status = L.device_status


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return L.CB_BF16
    if dt == torch.float32:
        return L.CB_F32
    raise ValueError(f"unsupported dtype {dt}")


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _s(stream=None):
    st = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(st.cuda_stream)


# ------------------------------------------------------------ primitives --
def cb_rope_table_init(max_positions: int, head_dim: int, rope_base: float,
                       device="cuda", stream=None) -> torch.Tensor:
    n = lib.cb_rope_table_elems(max_positions, head_dim)
    t = torch.empty(n, dtype=torch.float32, device=device)
    check(lib.cb_rope_table_init(_p(t), max_positions, head_dim,
                                 float(rope_base), _s(stream)))
    return t


def cb_rope_reposition(descs, layer_begin, layer_end, k_cache, v_cache,
                       cache_layer_stride, row_elems, head_dim, rope_table,
                       max_positions, stream=None):
    """descs: list of (k_src, v_src, src_layer_stride, len, dst_row, delta)
    with k_src / v_src torch tensors (their data pointers are used)."""
    arr = (L.StitchDesc * max(1, len(descs)))()
    for i, (ks, vs, stride, ln, dst, delta) in enumerate(descs):
        arr[i] = L.StitchDesc(ks.data_ptr(), vs.data_ptr(), stride, ln, dst, delta)
    check(lib.cb_rope_reposition(arr, len(descs), layer_begin, layer_end,
                                 _p(k_cache), _p(v_cache), cache_layer_stride,
                                 row_elems, head_dim, _p(rope_table),
                                 max_positions, dtype_code(k_cache.dtype),
                                 _s(stream)))


def cb_kv_deviation_topk(k_fresh, k_reused, reqs, policy, dev_out, idx_out,
                         ws=None, stream=None):
    """reqs: list of dicts with n_ctx, k, fresh_row0, reused_row0,
    dev_offset, idx_offset and (doc-aligned) span_offsets.  ws is reserved
    by the library (the selection needs no scratch) and may stay None."""
    n = len(reqs)
    arr, keep = _select_reqs(reqs)
    check(lib.cb_kv_deviation_topk(
        _p(k_fresh), k_fresh.stride(0), _p(k_reused), k_reused.stride(0),
        k_fresh.shape[1], dtype_code(k_fresh.dtype), arr, n, policy,
        _p(dev_out), _p(idx_out), _p(ws), 0 if ws is None else ws.numel(), _s(stream)))


def _select_reqs(reqs, dev_offsets=True):
    """ctypes cb_select_req array from dicts (n_ctx, k, fresh_row0,
    reused_row0, dev_offset, idx_offset, span_offsets, span_order, span_len,
    span_offset); the second value keeps the host arrays alive."""
    n = len(reqs)
    arr = (L.SelectReq * max(1, n))()
    keep = []

    def ints(v):
        if v is None:
            return None
        a = (C.c_int32 * max(1, len(v)))(*[int(x) for x in v])
        keep.append(a)
        return C.cast(a, C.POINTER(C.c_int32))
    for i, r in enumerate(reqs):
        spans = r.get("span_offsets")
        ns = len(spans) - 1 if spans is not None else 0
        arr[i] = L.SelectReq(r["n_ctx"], r["k"], r.get("fresh_row0", 0),
                             r.get("reused_row0", 0),
                             r.get("dev_offset", 0) if dev_offsets else 0,
                             r.get("idx_offset", 0), ns, ints(spans),
                             ints(r.get("span_order")), r.get("span_len", 0),
                             r.get("span_offset", 0))
    return arr, keep


def cb_kv_deviation_topk_noalloc(k_fresh, k_reused, reqs, policy, idx_out,
                                 stream=None):
    """cb_kv_deviation_topk without caller scratch: for callers that cannot
    allocate device memory, the deviations live in the library's fixed
    device array (at most 1048576 context tokens per call).  reqs as for
    cb_kv_deviation_topk; dev_offset is ignored."""
    n = len(reqs)
    arr, keep = _select_reqs(reqs, dev_offsets=False)
    check(lib.cb_kv_deviation_topk_noalloc(
        _p(k_fresh), k_fresh.stride(0), _p(k_reused), k_reused.stride(0),
        k_fresh.shape[1], dtype_code(k_fresh.dtype), arr, n, policy,
        _p(idx_out), _s(stream)))


def cb_gather_rows(src, idx, dst, stream=None):
    check(lib.cb_gather_rows(_p(src), src.stride(0), src.shape[0], _p(idx),
                             idx.numel(), src.shape[1], _p(dst), dst.stride(0),
                             dtype_code(src.dtype), _s(stream)))


def cb_scatter_kv(k_new, v_new, rows, k_cache, v_cache, stream=None):
    check(lib.cb_scatter_kv(_p(k_new), _p(v_new), k_new.stride(0), _p(rows),
                            rows.numel(), _p(k_cache), _p(v_cache),
                            k_cache.stride(0), k_cache.shape[0], k_new.shape[1],
                            dtype_code(k_new.dtype), _s(stream)))


def _attn_reqs(reqs):
    arr = (L.AttnReq * max(1, len(reqs)))()
    for i, (qb, qe, kv0, kvl) in enumerate(reqs):
        arr[i] = L.AttnReq(qb, qe, kv0, kvl)
    return arr


def cb_sparse_query_attention(q, q_pos, reqs, k_cache, v_cache, n_q_heads,
                              n_kv_heads, head_dim, out, scale=None, ws=None,
                              stream=None):
    """reqs: list of (q_begin, q_end, kv_row0, kv_len)."""
    scale = 1.0 / math.sqrt(head_dim) if scale is None else scale
    ar = _attn_reqs(reqs)
    need = lib.cb_attention_workspace_size(ar, len(reqs), n_q_heads, n_kv_heads,
                                           head_dim, dtype_code(q.dtype))
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    check(lib.cb_sparse_query_attention(
        _p(q), q.stride(0), _p(q_pos), ar, len(reqs),
        _p(k_cache), _p(v_cache), k_cache.stride(0), n_q_heads, n_kv_heads,
        head_dim, float(scale), _p(out), out.stride(0), dtype_code(q.dtype),
        _p(ws), ws.numel(), _s(stream)))


def cb_debug_expire_wait(limit_us: int, stream=None):
    check(lib.cb_debug_expire_wait(limit_us, _s(stream)))


def cb_debug_gemm_path(path: int):
    check(lib.cb_debug_gemm_path(path))


# ----------------------------------------------------------------- model --
@dataclass
class Seg:
    """A request segment: cached (k_pic/v_pic set) or recomputed."""
    len: int
    k_pic: torch.Tensor | None = None     # any tensor whose data_ptr() is
    v_pic: torch.Tensor | None = None     # the PIC base of this segment
    pic_layer_stride: int = 0
    pic_pos0: int = 0


@dataclass
class Req:
    tokens: torch.Tensor                  # device int32 [T]
    segs: list = field(default_factory=list)


def _requests(reqs):
    arr = (L.Request * len(reqs))()
    keep = []
    for i, r in enumerate(reqs):
        sa = (L.Segment * len(r.segs))()
        for j, s in enumerate(r.segs):
            sa[j] = L.Segment(s.len, None if s.k_pic is None else s.k_pic.data_ptr(),
                              None if s.v_pic is None else s.v_pic.data_ptr(),
                              s.pic_layer_stride, s.pic_pos0)
        keep.append(sa)
        arr[i] = L.Request(r.tokens.data_ptr(), C.cast(sa, C.POINTER(L.Segment)),
                           len(r.segs))
    return arr, keep


class BlendModel:
    """Device-resident weights plus the library's model handle."""

    def __init__(self, shape, dev_weights: dict, max_positions: int,
                 device="cuda"):
        self.shape = shape
        self.device = torch.device(device)
        self.dtype = torch_dtype(shape.dtype)
        self.w = dev_weights
        self.max_positions = max_positions
        self.rope_table = cb_rope_table_init(max_positions, shape.head_dim,
                                             shape.rope_base, device)
        cfg = L.ModelConfig(shape.n_layers, shape.d_model, shape.n_q_heads,
                            shape.n_kv_heads, shape.head_dim, shape.d_ffn,
                            shape.vocab, shape.rope_base, shape.norm_eps,
                            dtype_code(self.dtype), max_positions)
        self._layers = (L.LayerWeights * shape.n_layers)()
        for l, lw in enumerate(dev_weights["layers"]):
            self._layers[l] = L.LayerWeights(
                lw["w_qkv"].data_ptr(), lw["w_o"].data_ptr(),
                lw["w_gate"].data_ptr(), lw["w_up"].data_ptr(),
                lw["w_down"].data_ptr(), lw["norm1"].data_ptr(),
                lw["norm2"].data_ptr())
        wts = L.Weights(dev_weights["embed"].data_ptr(),
                        dev_weights["final_norm"].data_ptr(),
                        C.cast(self._layers, C.POINTER(L.LayerWeights)),
                        self.rope_table.data_ptr())
        h = C.c_void_p()
        check(lib.cb_model_create(C.byref(cfg), C.byref(wts), C.byref(h)))
        self.handle = h

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            lib.cb_model_destroy(h)
            self.handle = None

    # -------------------------------------------------------- construction
    @classmethod
    def from_host(cls, shape, weights: dict, max_positions: int,
                  device="cuda"):
        """Upload generator weights (float32 numpy arrays holding values of
        the model dtype) to the device."""
        dt = torch_dtype(shape.dtype)
        up = lambda a, d=dt: torch.from_numpy(np.ascontiguousarray(a)).to(
            device=device, dtype=d)
        dw = {"embed": up(weights["embed"]),
              "final_norm": up(weights["final_norm"], torch.float32),
              "layers": []}
        for lw in weights["layers"]:
            dw["layers"].append({
                "w_qkv": up(lw["w_qkv"]), "w_o": up(lw["w_o"]),
                "w_gate": up(lw["w_gate"]), "w_up": up(lw["w_up"]),
                "w_down": up(lw["w_down"]),
                "norm1": up(lw["norm1"], torch.float32),
                "norm2": up(lw["norm2"], torch.float32)})
        return cls(shape, dw, max_positions, device)

    @property
    def kvw(self):
        return self.shape.n_kv_heads * self.shape.head_dim

    # ------------------------------------------------------------- calls
    def cb_linear(self, A, W, out, epi=L.CB_EPI_STORE, W2=None, stream=None):
        M, K = A.shape
        N = W.shape[0]
        check(lib.cb_linear(self.handle, _p(A), A.stride(0), _p(W), _p(W2),
                            W.stride(0), M, N, K, epi, _p(out), out.stride(0),
                            _s(stream)))

    def cb_linear_ws(self, A, W, out, epi=L.CB_EPI_STORE, W2=None, ws=None, stream=None):
        """cb_linear with the tail-split workspace (allocated here when ws is None)."""
        M, K = A.shape
        N = W.shape[0]
        need = lib.cb_linear_workspace_size()
        if ws is None:
            ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        check(lib.cb_linear_ws(self.handle, _p(A), A.stride(0), _p(W), _p(W2),
                               W.stride(0), M, N, K, epi, _p(out), out.stride(0),
                               _p(ws), ws.numel() * ws.element_size(), _s(stream)))

    def cb_blend_layer(self, layer, h, pos, cache_row, reqs, k_cache, v_cache,
                       ws=None, stream=None):
        n = h.shape[0]
        need = lib.cb_layer_workspace_size(self.handle, n)
        if ws is None:
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        check(lib.cb_blend_layer(self.handle, layer, _p(h), n, _p(pos),
                                 _p(cache_row), _attn_reqs(reqs), len(reqs),
                                 _p(k_cache), _p(v_cache), _p(ws), ws.numel(),
                                 _s(stream)))

    def _params(self, ratio_bp, policy, sel_layer, schedule, forced=None, span_len=0,
                span_offset=0, span_order=None, query=None, forced_kept=None,
                host_load_ctas=0):
        """query: for the query-aware policies, a dict with anchor_rule,
        anchor_bp and crit_layers (QCFuse Eqs. 14, 20), and optionally
        anchors (a device int32 tensor in cb_anchor_select's layout: the
        chunks' precomputed anchors)."""
        n = len(schedule or [])
        sch = (L.ScheduleStep * max(1, n))()
        for i, (l, k) in enumerate(schedule or []):
            sch[i] = L.ScheduleStep(l, k)
        order = None
        if span_order is not None:
            order = (C.c_int32 * max(1, len(span_order)))(*[int(x) for x in span_order])
        q = query or {}
        crit = [int(x) for x in q.get("crit_layers", [])]
        crit_arr = (C.c_int32 * max(1, len(crit)))(*crit)
        return L.BlendParams(ratio_bp, policy, sel_layer, n,
                             C.cast(sch, C.POINTER(L.ScheduleStep)), span_len, span_offset,
                             None if order is None else C.cast(order, C.POINTER(C.c_int32)),
                             None if forced is None else forced.data_ptr(),
                             int(q.get("anchor_rule", L.CB_ANCHOR_SINK)),
                             int(q.get("anchor_bp", 0)), len(crit),
                             C.cast(crit_arr, C.POINTER(C.c_int32)),
                             None if forced_kept is None else forced_kept.data_ptr(),
                             int(host_load_ctas),
                             None if q.get("anchors") is None else q["anchors"].data_ptr()), \
            (sch, order, crit_arr)

    def plan(self, reqs, ratio_bp=None, policy=0, sel_layer=1, schedule=None, span_len=0,
             span_offset=0, span_order=None, query=None):
        arr, keep = _requests(reqs)
        out = L.Plan()
        if ratio_bp is None:
            check(lib.cb_full_plan(self.handle, arr, len(reqs), C.byref(out)))
        else:
            p, sch = self._params(ratio_bp, policy, sel_layer, schedule, None, span_len,
                                  span_offset, span_order, query)
            check(lib.cb_blend_plan(self.handle, arr, len(reqs), C.byref(p),
                                    C.byref(out)))
        return out

    def alloc_outputs(self, plan, B, blend=True):
        s = self.shape
        dev, dt = self.device, self.dtype
        T, N, K, R = plan.T_total, plan.N_total, plan.K_total, plan.R_total
        return {
            "k_cache": torch.empty(s.n_layers, T, self.kvw, dtype=dt, device=dev),
            "v_cache": torch.empty(s.n_layers, T, self.kvw, dtype=dt, device=dev),
            "deviation": torch.empty(max(N, 1), dtype=torch.float32, device=dev) if blend else None,
            "selected": torch.empty(max(K, 1), dtype=torch.int32, device=dev) if blend else None,
            "hidden": torch.empty(max(R, 1), s.d_model, dtype=torch.float32, device=dev),
            "rows": torch.empty(max(R, 1), dtype=torch.int32, device=dev),
            "first_token": torch.empty(B, dtype=torch.int32, device=dev),
            "workspace": torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev),
        }

    def _out(self, o, layer_stride=0):
        return L.BlendOut(o["k_cache"].data_ptr(), o["v_cache"].data_ptr(),
                          layer_stride,
                          None if o.get("deviation") is None else o["deviation"].data_ptr(),
                          None if o.get("selected") is None else o["selected"].data_ptr(),
                          None if o.get("hidden") is None else o["hidden"].data_ptr(),
                          None if o.get("rows") is None else o["rows"].data_ptr(),
                          None if o.get("first_token") is None else o["first_token"].data_ptr())

    def cb_blend_prefill(self, reqs, ratio_bp, policy=0, sel_layer=1,
                         schedule=None, outputs=None, forced=None,
                         stream=None, span_len=0, span_offset=0, span_order=None,
                         query=None, forced_kept=None):
        """forced: optional device int32 tensor of selected context
        positions (ascending per request) used instead of the ranking.
        forced_kept: with a schedule, the positions each gradual step keeps
        (device int32, step after step, requests in order) instead of its
        ranking.
        span_len / span_offset (fixed-chunk) and span_order (random-document,
        all requests' segment orders concatenated) as in cb_blend_params.
        query: anchor_rule / anchor_bp / crit_layers of the query-aware
        policies (sel_layer must then be 0)."""
        arr, keep = _requests(reqs)
        p, sch = self._params(ratio_bp, policy, sel_layer, schedule, forced, span_len,
                              span_offset, span_order, query, forced_kept)
        if outputs is None:
            plan = L.Plan()
            check(lib.cb_blend_plan(self.handle, arr, len(reqs), C.byref(p),
                                    C.byref(plan)))
            outputs = self.alloc_outputs(plan, len(reqs))
        o = self._out(outputs)
        ws = outputs["workspace"]
        check(lib.cb_blend_prefill(self.handle, arr, len(reqs), C.byref(p),
                                   C.byref(o), _p(ws), ws.numel(), _s(stream)))
        return outputs

    def cb_blend_prefill_host_kv(self, reqs, ratio_bp, copy_stream, policy=0, sel_layer=1,
                                 outputs=None, stream=None, span_len=0, span_offset=0,
                                 span_order=None, schedule=None, host_load_ctas=0,
                                 forced=None, query=None):
        """cb_blend_prefill with the requests' chunk caches in pinned host
        memory (HostChunkStore segments), loaded layer by layer on
        copy_stream while earlier layers compute.  host_load_ctas > 0: the
        re-position kernel reads the host caches directly with that many
        CTAs per layer (a bandwidth-bounded load) instead of the copy
        engines."""
        arr, keep = _requests(reqs)
        p, sch = self._params(ratio_bp, policy, sel_layer, schedule, forced, span_len,
                              span_offset, span_order, query=query,
                              host_load_ctas=host_load_ctas)
        if outputs is None:
            plan = L.Plan()
            check(lib.cb_blend_plan_host_kv(self.handle, arr, len(reqs), C.byref(p),
                                            C.byref(plan)))
            outputs = self.alloc_outputs(plan, len(reqs))
        o = self._out(outputs)
        ws = outputs["workspace"]
        check(lib.cb_blend_prefill_host_kv(self.handle, arr, len(reqs), C.byref(p),
                                           C.byref(o), _p(ws), ws.numel(), _s(stream),
                                           _s(copy_stream)))
        return outputs

    def cb_anchor_select(self, segs, rule, ratio_bp, with_scores=True, stream=None):
        """Per-chunk anchors of QCFuse Eq. 14 for cached segments (Seg):
        returns (anchors int32 [sum ceil(r_a |c|)], scores float [sum len] or
        None), chunk after chunk, chunk-local positions ascending."""
        sa = (L.Segment * len(segs))()
        for j, sg in enumerate(segs):
            sa[j] = L.Segment(sg.len, None if sg.k_pic is None else sg.k_pic.data_ptr(),
                              None if sg.v_pic is None else sg.v_pic.data_ptr(),
                              sg.pic_layer_stride, sg.pic_pos0)
        n_anchor = C.c_int64(0)
        check(lib.cb_anchor_count(sa, len(segs), ratio_bp, C.byref(n_anchor)))
        n_a = n_anchor.value
        n = sum(sg.len for sg in segs)
        anchors = torch.empty(max(n_a, 1), dtype=torch.int32, device=self.device)
        scores = torch.empty(max(n, 1), dtype=torch.float32, device=self.device) if with_scores else None
        need = lib.cb_anchor_workspace_size(self.handle, sa, len(segs))
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
        check(lib.cb_anchor_select(self.handle, sa, len(segs), rule, ratio_bp,
                                   None if scores is None else scores.data_ptr(),
                                   anchors.data_ptr(), _p(ws), ws.numel(), _s(stream)))
        return anchors[:n_a], (None if scores is None else scores[:n])

    def plan_host_kv(self, reqs, ratio_bp, policy=0, sel_layer=1, host_load_ctas=0, query=None):
        arr, keep = _requests(reqs)
        p, sch = self._params(ratio_bp, policy, sel_layer, None, query=query,
                              host_load_ctas=host_load_ctas)
        out = L.Plan()
        check(lib.cb_blend_plan_host_kv(self.handle, arr, len(reqs), C.byref(p), C.byref(out)))
        return out

    def cb_full_prefill(self, reqs, outputs=None, layer_stride=0, stream=None):
        arr, keep = _requests(reqs)
        if outputs is None:
            plan = L.Plan()
            check(lib.cb_full_plan(self.handle, arr, len(reqs), C.byref(plan)))
            outputs = self.alloc_outputs(plan, len(reqs), blend=False)
        o = self._out(outputs, layer_stride)
        ws = outputs["workspace"]
        check(lib.cb_full_prefill(self.handle, arr, len(reqs), C.byref(o),
                                  _p(ws), ws.numel(), _s(stream)))
        return outputs


class ChunkStore:
    """Per-chunk PIC caches kept in one device pool [n_layers][rows][kvw]
    (QCFuse Eq. 3: each chunk prefilled alone at positions 0..|c|-1).
    Chunks occupy runs of pool rows; evicted runs are reused first-fit, so a
    rolling window of equal-length documents cycles through fixed slots."""

    def __init__(self, model: BlendModel, capacity_rows: int):
        s = model.shape
        self.model = model
        self.capacity = capacity_rows
        self.K = torch.empty(s.n_layers, capacity_rows, model.kvw,
                             dtype=model.dtype, device=model.device)
        self.V = torch.empty_like(self.K)
        self.where = {}                      # chunk id -> (row, len)
        self.free = [(0, capacity_rows)]     # free row runs, ascending

    @property
    def used(self) -> int:
        return self.capacity - sum(n for _, n in self.free)

    def _alloc(self, n: int) -> int:
        for i, (r, m) in enumerate(self.free):
            if m >= n:
                if m == n:
                    self.free.pop(i)
                else:
                    self.free[i] = (r + n, m - n)
                return r
        raise RuntimeError("chunk store is full")

    def evict(self, cid):
        """Drops a chunk; its rows become free (merged with neighbours)."""
        r, n = self.where.pop(cid)
        runs = sorted(self.free + [(r, n)])
        merged = []
        for a, m in runs:
            if merged and merged[-1][0] + merged[-1][1] == a:
                merged[-1] = (merged[-1][0], merged[-1][1] + m)
            else:
                merged.append((a, m))
        self.free = merged

    def prefill(self, chunks: dict, stream=None):
        """chunks: {chunk_id: device int32 token tensor}; prefilled as one
        batch of standalone requests into one run of pool rows per batch."""
        items = list(chunks.items())
        for cid, _ in items:
            if cid in self.where:
                raise ValueError(f"chunk {cid!r} is already stored")
        for i in range(0, len(items), L.CB_MAX_BATCH):
            part = items[i:i + L.CB_MAX_BATCH]
            n = sum(int(t.numel()) for _, t in part)
            row0 = self._alloc(n)
            reqs = [Req(t, [Seg(int(t.numel()))]) for _, t in part]
            plan = self.model.plan(reqs)
            dev = self.model.device
            outs = {
                "k_cache": self.K[:, row0:],
                "v_cache": self.V[:, row0:],
                "hidden": None, "rows": None, "first_token": None,
                "workspace": torch.empty(max(plan.workspace_bytes, 256),
                                         dtype=torch.uint8, device=dev),
            }
            self.model.cb_full_prefill(reqs, outs,
                                       layer_stride=self.capacity * self.model.kvw,
                                       stream=stream)
            r = row0
            for cid, t in part:
                self.where[cid] = (r, int(t.numel()))
                r += int(t.numel())

    def seg(self, cid) -> Seg:
        r, n = self.where[cid]
        return Seg(n, self.K[0, r], self.V[0, r], self.capacity * self.model.kvw, 0)

    def write_back(self, items, outputs, stream=None):
        """Cache write-back ("Request Order Matters" §4.2, §5): replaces
        stored chunks by their fused K/V from a blended prefill, keys rotated
        back to chunk-local positions (cb_rope_reposition with a negative
        shift, all layers).  items: (chunk_id, fused-cache row of the chunk's
        first token, its request position); outputs: the prefill's outputs
        (k_cache / v_cache [n_layers][T_total][kvw])."""
        K, V = outputs["k_cache"], outputs["v_cache"]
        descs = []
        for cid, row, pos0 in items:
            r, n = self.where[cid]
            descs.append((K[0, row], V[0, row], K.stride(0), n, r, -int(pos0)))
        for i in range(0, len(descs), 64):
            cb_rope_reposition(descs[i:i + 64], 0, self.model.shape.n_layers, self.K, self.V,
                               self.capacity * self.model.kvw, self.model.kvw,
                               self.model.shape.head_dim, self.model.rope_table,
                               self.model.max_positions, stream)


class HostChunkStore:
    """Chunk caches kept in pinned host memory, [n_layers][rows][kvw] per K
    and V (the store CacheBlend loads from CPU memory or disk, "Hiding
    Recompute Behind I/O").  A chunk is prefilled standalone on the device
    (QCFuse Eq. 3) and its caches are copied to the host pool; requests use
    it through BlendModel.cb_blend_prefill_host_kv."""

    def __init__(self, model: BlendModel, capacity_rows: int):
        s = model.shape
        self.model = model
        self.capacity = capacity_rows
        self.K = torch.empty(s.n_layers, capacity_rows, model.kvw, dtype=model.dtype).pin_memory()
        self.V = torch.empty_like(self.K).pin_memory()
        self.where = {}
        self.used = 0

    def prefill(self, chunks: dict, stream=None):
        """chunks: {chunk_id: device int32 tokens}; computed on the device,
        then copied to the host pool (not part of a request's TTFT)."""
        n = sum(int(t.numel()) for t in chunks.values())
        if self.used + n > self.capacity:
            raise RuntimeError("host chunk store is full")
        tmp = ChunkStore(self.model, n)
        tmp.prefill(chunks, stream)
        torch.cuda.synchronize()
        for cid, t in chunks.items():
            r, m = tmp.where[cid]
            self.K[:, self.used:self.used + m].copy_(tmp.K[:, r:r + m])
            self.V[:, self.used:self.used + m].copy_(tmp.V[:, r:r + m])
            self.where[cid] = (self.used, m)
            self.used += m
        del tmp

    def seg(self, cid) -> Seg:
        r, n = self.where[cid]
        return Seg(n, self.K[0, r], self.V[0, r], self.capacity * self.model.kvw, 0)


def loading_controller(load_ms_per_layer: float, compute_ms_per_layer: dict,
                       min_ratio_bp: int = 1500) -> int:
    """cb_loading_ratio ([CB] "Hiding Recompute Behind I/O": r = max(r_load,
    15%)): compute_ms_per_layer is {ratio_bp: measured recompute ms per
    layer}; returns the ratio in basis points."""
    items = sorted(compute_ms_per_layer.items())
    n = len(items)
    ratios = (C.c_int32 * max(1, n))(*[int(r) for r, _ in items])
    times = (C.c_double * max(1, n))(*[float(t) for _, t in items])
    out = C.c_int32(0)
    check(lib.cb_loading_ratio(float(load_ms_per_layer), ratios, times, n, int(min_ratio_bp),
                               C.byref(out)))
    return out.value


class RollingWindow:
    """Serving loop of a rolling-agent window ("Request Order Matters" §4.1):
    every request holds the window's documents and a query.  The documents
    already seen are cached chunks in a persistent store; the newest one has
    no cache when its request is evaluated, so it is recomputed as an
    uncached segment.  After the request it is prefilled into the store and
    the oldest document is evicted (stride 1)."""

    def __init__(self, model: BlendModel, window: int, doc_rows: int,
                 ratio_bp: int, policy: int = L.CB_POLICY_DOC_ALIGNED,
                 write_back: bool = False):
        self.model = model
        self.write_back = write_back      # store each request's fused caches back
        self.window = window
        self.ratio_bp = ratio_bp
        self.policy = policy
        # the window's cached documents plus the one being added
        self.store = ChunkStore(model, (window + 1) * doc_rows)
        self.docs = []        # cached document ids, window order
        self.tokens = {}      # id -> device int32 tokens

    def seed(self, docs: dict, stream=None):
        """Prefills the documents that precede the first request."""
        self.store.prefill(docs, stream)
        for cid, t in docs.items():
            self.docs.append(cid)
            self.tokens[cid] = t

    def request(self, new_tokens, query_tokens):
        """The request for the current window plus one new document."""
        segs = [self.store.seg(c) for c in self.docs]
        segs += [Seg(int(new_tokens.numel())), Seg(int(query_tokens.numel()))]
        toks = torch.cat([self.tokens[c] for c in self.docs] + [new_tokens, query_tokens])
        return Req(toks.to(torch.int32).contiguous(), segs)

    def blend(self, req, outputs=None, stream=None, **span_args):
        """span_args: span_len / span_offset / span_order of cb_blend_params.
        With write_back, the cached documents' fused K/V replace their
        stored caches afterwards (the store then depends on history)."""
        out = self.model.cb_blend_prefill([req], self.ratio_bp, self.policy,
                                          outputs=outputs, stream=stream, **span_args)
        if self.write_back:
            items, pos = [], 0
            for cid in self.docs:
                items.append((cid, pos, pos))
                pos += self.store.where[cid][1]
            self.store.write_back(items, out, stream)
        return out

    def advance(self, new_id, new_tokens, stream=None):
        """Stores the new document's chunk cache; evicts the oldest once the
        window is full."""
        self.store.prefill({new_id: new_tokens}, stream)
        self.docs.append(new_id)
        self.tokens[new_id] = new_tokens
        if len(self.docs) > self.window - 1:
            old = self.docs.pop(0)
            self.store.evict(old)
            del self.tokens[old]


def selection_stats(selected: torch.Tensor, deviation: torch.Tensor, stream=None):
    """Diagnostics of one request's selection ("Request Order Matters" §4.4,
    Table 2), computed by cb_selection_stats: the number of contiguous
    regions it occupies and the share of the total deviation it carries.
    selected: ascending positions (device int32); deviation: d over the
    request's reusable tokens (device float).  Returns host values."""
    seg = torch.empty(1, dtype=torch.int32, device=deviation.device)
    cap = torch.empty(1, dtype=torch.float64, device=deviation.device)
    arr, keep = _select_reqs([dict(n_ctx=int(deviation.numel()), k=int(selected.numel()))])
    check(lib.cb_selection_stats(_p(deviation), _p(selected), arr, 1, _p(seg), _p(cap),
                                 _s(stream)))
    return int(seg.item()), float(cap.item())
