"""The C ABI used from C alone: tests/c_abi_blend.c, compiled here with gcc
against include/cacheblend.h, libcacheblend.so and the CUDA runtime,
prefills three chunks on their own and blends a request over them (fp32
model, 15% token top-k).  No Python or PyTorch is on its path.  Its
selection, computed rows, hidden states and first token must equal those of
the same calls made through the Python binding, bit for bit (the fp32 path
is deterministic and computes every row independently of the batch)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workload as W
import rag_kv_cache_layer_gb300 as R
from rag_kv_cache_layer_gb300 import _lib as L

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.isdir(os.path.join(cand, "include")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def _build(tmp_path):
    gcc, cuda = shutil.which("gcc"), _cuda_home()
    if not gcc or not cuda:
        pytest.skip("gcc or the CUDA toolkit is not available")
    lib_dir = os.path.dirname(L.LIB_PATH)
    libs = [d for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
            if os.path.exists(os.path.join(cuda, d, "libcudart.so"))]
    if not libs:
        pytest.skip("libcudart.so not found")
    cudart = os.path.join(cuda, libs[0])
    exe = str(tmp_path / "c_abi_blend")
    subprocess.run([gcc, "-O2", "-std=c11", "-Wall", "-o", exe,
                    os.path.join(HERE, "c_abi_blend.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", lib_dir, "-lcacheblend", "-L", cudart, "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cudart}"],
                   check=True, capture_output=True, text=True)
    return exe


def _write_input(path, shape, weights, chunks, query, ratio_bp, max_pos):
    with open(path, "wb") as f:
        np.array([shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads,
                  shape.head_dim, shape.d_ffn, shape.vocab, max_pos, len(chunks), len(query),
                  ratio_bp], np.int32).tofile(f)
        np.array([shape.rope_base, shape.norm_eps], np.float32).tofile(f)
        np.array([len(c) for c in chunks], np.int32).tofile(f)
        np.asarray(weights["embed"], np.float32).tofile(f)
        np.asarray(weights["final_norm"], np.float32).tofile(f)
        for lw in weights["layers"]:
            for key in ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "norm1", "norm2"):
                np.ascontiguousarray(lw[key], np.float32).tofile(f)
        np.concatenate(list(chunks) + [query]).astype(np.int32).tofile(f)


def test_blend_driven_from_c_matches_the_binding(tmp_path):
    exe = _build(tmp_path)
    shape, max_pos, ratio_bp = W.TINY_F32, 1024, 1500
    rng = np.random.default_rng(21)
    weights = W.make_weights(shape, 17)
    chunks = [W.make_tokens(rng, n, shape.vocab) for n in (128, 75, 200)]
    query = W.make_tokens(rng, 23, shape.vocab)
    inp, outp = str(tmp_path / "in.bin"), str(tmp_path / "out.bin")
    _write_input(inp, shape, weights, chunks, query, ratio_bp, max_pos)
    run = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr

    raw = np.fromfile(outp, np.int32)
    K, Rn, first = (int(x) for x in raw[:3])
    sel_c = raw[3:3 + K]
    rows_c = raw[3 + K:3 + K + Rn]
    hidden_c = raw[3 + K + Rn:].view(np.float32).reshape(Rn, shape.d_model)

    model = R.BlendModel.from_host(shape, weights, max_pos)
    store = R.ChunkStore(model, sum(len(c) for c in chunks))
    store.prefill({i: torch.from_numpy(c).cuda() for i, c in enumerate(chunks)})
    toks = torch.from_numpy(np.concatenate(chunks + [query]).astype(np.int32)).cuda()
    req = R.Req(toks, [store.seg(i) for i in range(len(chunks))] + [R.Seg(len(query))])
    out = model.cb_blend_prefill([req], ratio_bp)
    torch.cuda.synchronize()
    assert R.device_status() == 0
    assert K == len(sel_c) and K > 0
    assert np.array_equal(sel_c, out["selected"][:K].cpu().numpy())
    assert np.array_equal(rows_c, out["rows"][:Rn].cpu().numpy())
    assert np.array_equal(hidden_c, out["hidden"][:Rn].cpu().numpy())
    assert first == int(out["first_token"][0])
