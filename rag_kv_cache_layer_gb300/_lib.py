"""ctypes binding of libcacheblend.so (the C ABI in include/cacheblend.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Importing this module loads the shared library and raises if it is
missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcacheblend.so")

# status codes / enums (include/cacheblend.h)
CB_OK, CB_ERR_INVALID_ARG, CB_ERR_UNSUPPORTED, CB_ERR_CUDA, CB_ERR_TIMEOUT, \
    CB_ERR_DEVICE_INDEX, CB_ERR_WORKSPACE = range(7)
STATUS_NAMES = {0: "CB_OK", 1: "CB_ERR_INVALID_ARG", 2: "CB_ERR_UNSUPPORTED",
                3: "CB_ERR_CUDA", 4: "CB_ERR_TIMEOUT", 5: "CB_ERR_DEVICE_INDEX",
                6: "CB_ERR_WORKSPACE"}
CB_F32, CB_BF16 = 0, 1
CB_POLICY_TOKEN_TOPK, CB_POLICY_DOC_ALIGNED = 0, 1
CB_POLICY_SINGLE_WINDOW, CB_POLICY_FIXED_CHUNK, CB_POLICY_RANDOM_DOC = 2, 3, 4
CB_POLICY_FIRST_TOKENS = 5
CB_POLICY_QUERY_PROBE, CB_POLICY_QUERY_FULL = 6, 7
CB_ANCHOR_SINK, CB_ANCHOR_KNORM = 0, 1
CB_EPI_STORE, CB_EPI_RESID, CB_EPI_SWIGLU = 0, 1, 2
CB_GEMM_AUTO, CB_GEMM_TOKEN_M, CB_GEMM_SWAP_AB, CB_GEMM_SWAP_AB_PAIR = 0, 1, 2, 3
CB_PROBE_QKV, CB_PROBE_O, CB_PROBE_SWIGLU, CB_PROBE_DOWN, CB_PROBE_ATTENTION = 1, 2, 3, 4, 5
CB_PROBE_STITCH, CB_PROBE_SELECT, CB_PROBE_GATHER, CB_PROBE_LM_HEAD = 6, 7, 8, 9
CB_PROBE_MLP = 10
CB_MAX_BATCH = 64
CB_MAX_SPANS = 1024


class CBError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


vp = C.c_void_p
i32 = C.c_int
i64 = C.c_int64


class StitchDesc(C.Structure):
    _fields_ = [("k_src", vp), ("v_src", vp), ("src_layer_stride", i64),
                ("len", i32), ("dst_row", i32), ("delta", i32)]


class SelectReq(C.Structure):
    _fields_ = [("n_ctx", i32), ("k", i32), ("fresh_row0", i64),
                ("reused_row0", i64), ("dev_offset", i32), ("idx_offset", i32),
                ("n_spans", i32), ("span_offsets", C.POINTER(C.c_int32)),
                ("span_order", C.POINTER(C.c_int32)), ("span_len", i32),
                ("span_offset", i32)]


class AttnReq(C.Structure):
    _fields_ = [("q_begin", i32), ("q_end", i32), ("kv_row0", i64),
                ("kv_len", i32)]


class ModelConfig(C.Structure):
    _fields_ = [("n_layers", i32), ("d_model", i32), ("n_q_heads", i32),
                ("n_kv_heads", i32), ("head_dim", i32), ("d_ffn", i32),
                ("vocab", i32), ("rope_base", C.c_float),
                ("norm_eps", C.c_float), ("dtype", i32),
                ("max_positions", i32)]


class LayerWeights(C.Structure):
    _fields_ = [("w_qkv", vp), ("w_o", vp), ("w_gate", vp), ("w_up", vp),
                ("w_down", vp), ("norm1", vp), ("norm2", vp)]


class Weights(C.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp),
                ("layers", C.POINTER(LayerWeights)), ("rope_table", vp)]


class Segment(C.Structure):
    _fields_ = [("len", i32), ("k_pic", vp), ("v_pic", vp),
                ("pic_layer_stride", i64), ("pic_pos0", i32)]


class Request(C.Structure):
    _fields_ = [("tokens", vp), ("segments", C.POINTER(Segment)),
                ("n_segments", i32)]


class ScheduleStep(C.Structure):
    _fields_ = [("layer", i32), ("keep", i32)]


class BlendParams(C.Structure):
    _fields_ = [("ratio_bp", i32), ("policy", i32), ("sel_layer", i32),
                ("n_schedule", i32), ("schedule", C.POINTER(ScheduleStep)),
                ("span_len", i32), ("span_offset", i32),
                ("span_order", C.POINTER(C.c_int32)), ("forced_selected", vp),
                ("anchor_rule", i32), ("anchor_bp", i32), ("n_crit", i32),
                ("crit_layers", C.POINTER(C.c_int32)), ("forced_kept", vp),
                ("host_load_ctas", i32), ("anchors", vp)]


class BlendOut(C.Structure):
    _fields_ = [("k_cache", vp), ("v_cache", vp), ("cache_layer_stride", i64),
                ("deviation", vp), ("selected", vp), ("hidden", vp),
                ("rows", vp), ("first_token", vp)]


class Plan(C.Structure):
    _fields_ = [("T_total", i64), ("N_total", i64), ("K_total", i64),
                ("R_total", i64), ("workspace_bytes", C.c_size_t),
                ("K_final", i64), ("R_final", i64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python rag_kv_cache_layer_gb300/build.py` (there is no CPU path)")
    lib = C.CDLL(LIB_PATH)
    S = i32  # cb_status
    sigs = {
        "cb_last_error_message": (C.c_char_p, []),
        "cb_version": (i32, []),
        "cb_get_device_status": (S, [C.POINTER(i32)]),
        "cb_debug_expire_wait": (S, [i32, vp]),
        "cb_debug_launch_count": (C.c_ulonglong, []),
        "cb_debug_gemm_path": (S, [i32]),
        "cb_debug_index_checks": (S, [i32]),
        "cb_debug_mlp_fusion": (S, [i32]),
        "cb_debug_mlp_one_launch": (i32, [i32, i32, i32]),
        "cb_debug_probe_start": (S, [i32, i32]),
        "cb_debug_probe_stop": (S, [C.POINTER(i32), C.POINTER(C.c_float)]),
        "cb_rope_table_elems": (C.c_size_t, [i32, i32]),
        "cb_rope_table_init": (S, [vp, i32, i32, C.c_float, vp]),
        "cb_rope_reposition": (S, [C.POINTER(StitchDesc), i32, i32, i32, vp, vp,
                                   i64, i32, i32, vp, i32, i32, vp]),
        "cb_select_workspace_size": (C.c_size_t, [i32]),
        "cb_kv_deviation_topk": (S, [vp, i64, vp, i64, i32, i32,
                                     C.POINTER(SelectReq), i32, i32, vp, vp, vp,
                                     C.c_size_t, vp]),
        "cb_kv_deviation_topk_noalloc": (S, [vp, i64, vp, i64, i32, i32,
                                             C.POINTER(SelectReq), i32, i32, vp, vp]),
        "cb_gather_rows": (S, [vp, i64, i64, vp, i32, i32, vp, i64, i32, vp]),
        "cb_scatter_kv": (S, [vp, vp, i64, vp, i32, vp, vp, i64, i64, i32, i32, vp]),
        "cb_attention_workspace_size": (C.c_size_t, [C.POINTER(AttnReq), i32, i32,
                                                     i32, i32, i32]),
        "cb_sparse_query_attention": (S, [vp, i64, vp, C.POINTER(AttnReq), i32,
                                          vp, vp, i64, i32, i32, i32, C.c_float,
                                          vp, i64, i32, vp, C.c_size_t, vp]),
        "cb_model_create": (S, [C.POINTER(ModelConfig), C.POINTER(Weights),
                                C.POINTER(vp)]),
        "cb_model_destroy": (None, [vp]),
        "cb_linear": (S, [vp, vp, i64, vp, vp, i64, i32, i32, i32, i32, vp, i64, vp]),
        "cb_linear_workspace_size": (C.c_size_t, []),
        "cb_linear_ws": (S, [vp, vp, i64, vp, vp, i64, i32, i32, i32, i32, vp, i64, vp,
                             C.c_size_t, vp]),
        "cb_blend_plan": (S, [vp, C.POINTER(Request), i32, C.POINTER(BlendParams),
                              C.POINTER(Plan)]),
        "cb_blend_prefill": (S, [vp, C.POINTER(Request), i32,
                                 C.POINTER(BlendParams), C.POINTER(BlendOut), vp,
                                 C.c_size_t, vp]),
        "cb_blend_plan_host_kv": (S, [vp, C.POINTER(Request), i32, C.POINTER(BlendParams),
                                      C.POINTER(Plan)]),
        "cb_blend_prefill_host_kv": (S, [vp, C.POINTER(Request), i32,
                                         C.POINTER(BlendParams), C.POINTER(BlendOut), vp,
                                         C.c_size_t, vp, vp]),
        "cb_full_plan": (S, [vp, C.POINTER(Request), i32, C.POINTER(Plan)]),
        "cb_full_prefill": (S, [vp, C.POINTER(Request), i32, C.POINTER(BlendOut),
                                vp, C.c_size_t, vp]),
        "cb_layer_workspace_size": (C.c_size_t, [vp, i32]),
        "cb_blend_layer": (S, [vp, i32, vp, i32, vp, vp, C.POINTER(AttnReq), i32,
                               vp, vp, vp, C.c_size_t, vp]),
        "cb_anchor_workspace_size": (C.c_size_t, [vp, C.POINTER(Segment), i32]),
        "cb_anchor_select": (S, [vp, C.POINTER(Segment), i32, i32, i32, vp, vp, vp,
                                 C.c_size_t, vp]),
        "cb_anchor_count": (S, [C.POINTER(Segment), i32, i32, C.POINTER(i64)]),
        "cb_loading_ratio": (S, [C.c_double, C.POINTER(C.c_int32), C.POINTER(C.c_double), i32,
                                 C.c_int32, C.POINTER(C.c_int32)]),
        "cb_selection_stats": (S, [vp, vp, C.POINTER(SelectReq), i32, vp, vp, vp]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()

# names every build of the library must export (include/cacheblend.h)
EXPORTED = [
    "cb_last_error_message", "cb_version", "cb_get_device_status",
    "cb_debug_expire_wait", "cb_debug_launch_count", "cb_debug_gemm_path",
    "cb_debug_index_checks", "cb_debug_mlp_fusion", "cb_debug_mlp_one_launch",
    "cb_debug_probe_start", "cb_debug_probe_stop",
    "cb_rope_table_elems",
    "cb_rope_table_init",
    "cb_rope_reposition", "cb_select_workspace_size", "cb_kv_deviation_topk",
    "cb_kv_deviation_topk_noalloc",
    "cb_gather_rows", "cb_scatter_kv", "cb_attention_workspace_size",
    "cb_sparse_query_attention",
    "cb_model_create", "cb_model_destroy", "cb_linear", "cb_linear_workspace_size",
    "cb_linear_ws", "cb_blend_plan",
    "cb_blend_prefill", "cb_blend_plan_host_kv", "cb_blend_prefill_host_kv",
    "cb_full_plan", "cb_full_prefill",
    "cb_layer_workspace_size", "cb_blend_layer",
    "cb_anchor_workspace_size", "cb_anchor_select", "cb_anchor_count",
    "cb_loading_ratio", "cb_selection_stats",
]


def check(status: int) -> None:
    if status != CB_OK:
        raise CBError(status, lib.cb_last_error_message().decode())


def device_status() -> int:
    """Reads and clears the device status word (synchronises the device)."""
    out = i32(0)
    check(lib.cb_get_device_status(C.byref(out)))
    return out.value
