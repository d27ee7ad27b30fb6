"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, its ctypes mirrors match the C struct layouts, and host-side
validation rejects bad arguments before anything touches a device."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cacheblend.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cb_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_entry_point_is_exported():
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L.lib, n), n
    assert sorted(L.EXPORTED) == sorted(n for n in names if n in L.EXPORTED)
    assert set(names) <= set(L.EXPORTED) | set(getattr(L, "EXTRA_EXPORTED", []))


STRUCTS = {
    "cb_stitch_desc": (L.StitchDesc, ["k_src", "v_src", "src_layer_stride", "len", "dst_row", "delta"]),
    "cb_select_req": (L.SelectReq, ["n_ctx", "k", "fresh_row0", "reused_row0", "dev_offset",
                                    "idx_offset", "n_spans", "span_offsets", "span_order",
                                    "span_len", "span_offset"]),
    "cb_attn_req": (L.AttnReq, ["q_begin", "q_end", "kv_row0", "kv_len"]),
    "cb_model_config": (L.ModelConfig, ["n_layers", "d_model", "n_q_heads", "n_kv_heads",
                                        "head_dim", "d_ffn", "vocab", "rope_base", "norm_eps",
                                        "dtype", "max_positions"]),
    "cb_layer_weights": (L.LayerWeights, ["w_qkv", "w_o", "w_gate", "w_up", "w_down",
                                          "norm1", "norm2"]),
    "cb_weights": (L.Weights, ["embed", "final_norm", "layers", "rope_table"]),
    "cb_segment": (L.Segment, ["len", "k_pic", "v_pic", "pic_layer_stride", "pic_pos0"]),
    "cb_request": (L.Request, ["tokens", "segments", "n_segments"]),
    "cb_schedule_step": (L.ScheduleStep, ["layer", "keep"]),
    "cb_blend_params": (L.BlendParams, ["ratio_bp", "policy", "sel_layer", "n_schedule",
                                        "schedule", "span_len", "span_offset", "span_order",
                                        "forced_selected", "anchor_rule", "anchor_bp",
                                        "n_crit", "crit_layers", "forced_kept",
                                        "host_load_ctas"]),
    "cb_blend_out": (L.BlendOut, ["k_cache", "v_cache", "cache_layer_stride", "deviation",
                                  "selected", "hidden", "rows", "first_token"]),
    "cb_plan": (L.Plan, ["T_total", "N_total", "K_total", "R_total", "workspace_bytes",
                         "K_final", "R_final"]),
}


def test_ctypes_mirrors_match_c_layout():
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "cacheblend.h"',
             "int main(void) {"]
    for cname, (_, fields) in STRUCTS.items():
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for f in fields:
            lines.append(f'  printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("  return 0; }")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(src, "w").write("\n".join(lines))
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), src, "-o", exe],
                       check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    for cname, (ct, fields) in STRUCTS.items():
        assert int(got[cname]) == C.sizeof(ct), cname
        for f in fields:
            assert int(got[f"{cname}.{f}"]) == getattr(ct, f).offset, (cname, f)


def test_host_validation_without_device():
    lib = L.lib
    assert lib.cb_version() >= 100
    assert lib.cb_rope_table_elems(0, 64) == 0
    assert lib.cb_rope_table_elems(10, 64) == 640
    # NULL pointers are rejected before any CUDA call
    st = lib.cb_kv_deviation_topk(None, 0, None, 0, 64, L.CB_F32, None, 0, 0,
                                  None, None, None, 0, None)
    assert st == L.CB_ERR_INVALID_ARG
    assert "NULL" in lib.cb_last_error_message().decode()
    assert lib.cb_rope_table_init(None, 10, 64, 1e4, None) == L.CB_ERR_INVALID_ARG
    assert lib.cb_gather_rows(None, 0, 0, None, 0, 0, None, 0, 0, None) == L.CB_OK
    h = C.c_void_p()
    assert lib.cb_model_create(None, None, C.byref(h)) == L.CB_ERR_INVALID_ARG
    cfg = L.ModelConfig(2, 256, 4, 2, 48, 688, 4096, 1e4, 1e-5, 0, 1024)
    w = L.Weights(None, None, None, None)
    assert lib.cb_model_create(C.byref(cfg), C.byref(w), C.byref(h)) == L.CB_ERR_UNSUPPORTED
    assert lib.cb_debug_expire_wait(-1, None) == L.CB_ERR_INVALID_ARG
    assert lib.cb_debug_gemm_path(4) == L.CB_ERR_INVALID_ARG
    assert lib.cb_debug_gemm_path(L.CB_GEMM_AUTO) == L.CB_OK
    assert lib.cb_debug_probe_start(0, 4) == L.CB_ERR_INVALID_ARG
    assert lib.cb_debug_probe_start(L.CB_PROBE_SWIGLU, 0) == L.CB_ERR_INVALID_ARG
    assert lib.cb_debug_probe_start(L.CB_PROBE_MLP + 1, 4) == L.CB_ERR_INVALID_ARG
    assert lib.cb_debug_probe_stop(None, None) == L.CB_ERR_INVALID_ARG
    # anchors: NULL model / chunks / output, bad rule or ratio
    assert lib.cb_anchor_select(None, None, 1, 0, 1000, None, None, None, 0, None) == \
        L.CB_ERR_INVALID_ARG
    # bad doc-aligned spans are rejected on the host
    spans = (C.c_int32 * 3)(0, 5, 4)
    req = L.SelectReq(4, 2, 0, 0, 0, 0, 2, C.cast(spans, C.POINTER(C.c_int32)), None, 0, 0)
    ws = C.create_string_buffer(4096)
    st = lib.cb_kv_deviation_topk(C.c_void_p(16), 64, C.c_void_p(16), 64, 64, L.CB_F32,
                                  C.byref(req), 1, L.CB_POLICY_DOC_ALIGNED, C.c_void_p(16),
                                  C.c_void_p(16), ws, 4096, None)
    assert st == L.CB_ERR_INVALID_ARG


def test_span_policy_requests_are_validated_on_the_host():
    """Malformed span-policy requests fail before anything is enqueued
    (no GPU needed): a random-document order that is not a permutation or
    is missing, fixed chunks without a length or with an offset past it, and
    an unknown policy."""
    lib = L.lib
    ws = C.create_string_buffer(4096)
    spans = (C.c_int32 * 3)(0, 5, 10)
    sp = C.cast(spans, C.POINTER(C.c_int32))
    dup = (C.c_int32 * 2)(1, 1)
    cases = [
        (L.CB_POLICY_RANDOM_DOC, L.SelectReq(10, 3, 0, 0, 0, 0, 2, sp,
                                             C.cast(dup, C.POINTER(C.c_int32)), 0, 0)),
        (L.CB_POLICY_RANDOM_DOC, L.SelectReq(10, 3, 0, 0, 0, 0, 2, sp, None, 0, 0)),
        (L.CB_POLICY_FIXED_CHUNK, L.SelectReq(10, 3, 0, 0, 0, 0, 0, None, None, 0, 0)),
        (L.CB_POLICY_FIXED_CHUNK, L.SelectReq(10, 3, 0, 0, 0, 0, 0, None, None, 4, 5)),
        (7, L.SelectReq(10, 3, 0, 0, 0, 0, 2, sp, None, 0, 0)),
    ]
    for policy, req in cases:
        st = lib.cb_kv_deviation_topk(C.c_void_p(16), 64, C.c_void_p(16), 64, 64, L.CB_F32,
                                      C.byref(req), 1, policy, C.c_void_p(16), C.c_void_p(16),
                                      ws, 4096, None)
        assert st == L.CB_ERR_INVALID_ARG, policy
        assert lib.cb_last_error_message()


def test_loading_controller_rule():
    """[CB] "Hiding Recompute Behind I/O": r = max(r_load, 15%), r_load the
    largest measured ratio whose per-layer recompute fits in the per-layer
    load (host-only call)."""
    table = {500: 0.2, 1500: 0.25, 3000: 0.4, 5000: 0.6, 10000: 1.1}
    assert R.loading_controller(0.07, table) == 1500        # every load hides: the floor
    assert R.loading_controller(0.45, table) == 3000
    assert R.loading_controller(0.6, table) == 5000          # equal time still hides
    assert R.loading_controller(2.6, table) == 10000         # slow storage: recompute all
    assert R.loading_controller(0.45, table, min_ratio_bp=5000) == 5000
    import ctypes as C
    out = C.c_int32(0)
    bad = (C.c_int32 * 1)(10001)
    t = (C.c_double * 1)(0.1)
    assert L.lib.cb_loading_ratio(1.0, bad, t, 1, 1500, C.byref(out)) == L.CB_ERR_INVALID_ARG
    assert L.lib.cb_loading_ratio(float("nan"), None, None, 0, 1500, C.byref(out)) == L.CB_ERR_INVALID_ARG


def test_anchor_count_is_the_ceiling_per_chunk():
    """QCFuse Eq. 14: ceil(r_a |c_i|) anchors per chunk (host-only call)."""
    import ctypes as C
    segs = (L.Segment * 3)(L.Segment(512, None, None, 0, 0), L.Segment(7, None, None, 0, 0),
                           L.Segment(0, None, None, 0, 0))
    n = C.c_int64(0)
    L.check(L.lib.cb_anchor_count(segs, 3, 1000, C.byref(n)))
    assert n.value == 52 + 1 + 0
    L.check(L.lib.cb_anchor_count(segs, 3, 10000, C.byref(n)))
    assert n.value == 519
    assert L.lib.cb_anchor_count(segs, 3, 10001, C.byref(n)) == L.CB_ERR_INVALID_ARG


def test_debug_index_checks_switch_is_validated():
    assert L.lib.cb_debug_index_checks(2) == L.CB_ERR_INVALID_ARG
    L.check(L.lib.cb_debug_index_checks(1))
    L.check(L.lib.cb_debug_index_checks(0))


def test_debug_mlp_fusion_switch_is_validated():
    assert L.lib.cb_debug_mlp_fusion(2) == L.CB_ERR_INVALID_ARG
    assert L.lib.cb_debug_mlp_fusion(-1) == L.CB_ERR_INVALID_ARG
    L.check(L.lib.cb_debug_mlp_fusion(0))
    L.check(L.lib.cb_debug_mlp_fusion(1))
