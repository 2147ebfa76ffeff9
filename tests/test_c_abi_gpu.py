"""The prologue run from a C program on the GPU.

tests/c/prologue_gpu.c is a C99 caller that allocates device memory with its own
CUDA runtime and makes the calls a C user makes: row_quantize_e4m3 on the bf16
hidden state, the weight packing, qkv_cte_mx, kv_rms_norm_rope_cache and the
status readers.  This test writes a seeded problem to files, builds and runs that
program, and compares what it wrote back with the oracle: the activation codes
and scales bit for bit, the projection within the bf16 tolerance, and the int8
caches by the cache rules.
"""
import os
import shutil
import subprocess
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from parity_util import as_f64, check_kv, check_qkv, qkv_reference
from rope_attention_gb300 import build, synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


def _cuda_root():
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime_api.h")):
            return root
    return None


def _cudart_dir(root):
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return None


def test_prologue_from_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    root = _cuda_root()
    libcudart = _cudart_dir(root) if root else None
    if cc is None or libcudart is None:
        pytest.skip("no C compiler or CUDA runtime library")
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "prologue_gpu")
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-O2", "-I", INCLUDE,
           "-isystem", os.path.join(root, "include"), os.path.join(HERE, "c", "prologue_gpu.c"), "-o", exe,
           "-L", libdir, "-lrope_attention", f"-Wl,-rpath,{libdir}", "-L", libcudart, "-lcudart",
           f"-Wl,-rpath,{libcudart}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"

    # (a) a small self-attention layer: 300 tokens, H 256, 4 + 2 + 2 heads of 64
    S, H, nq, nkv, d = 300, 256, 4, 2, 64
    qc = synth.make_qkv("c_prologue", 81, S=S, H=H, num_heads=nq, num_kv_heads=nkv, head_dim=d)
    hidden = synth.hidden_bf16(82, S, H)
    # (b) the separate-kv KV call: V2, int8 per-head quantisation, PA_BNSD
    kc = synth.make_kv("c_prologue_kv", 83, variant=2, B=2, N=4, S=50, Dkv=192, Dv=128, block_size=32,
                       block_num=4, quant_k=True, quant_v=True, is_output_kv=False, skip_frac=0.1)
    files = {"hidden.bin": hidden, "w.bin": qc.w, "w_exp.bin": qc.w_block_exp, "bias.bin": qc.bias,
             "cos_q.bin": qc.cos.astype(np.float32), "sin_q.bin": qc.sin.astype(np.float32),
             "q_gamma.bin": qc.q_gamma, "k_gamma.bin": qc.k_gamma,
             "kv.bin": kc.kv, "v.bin": kc.v, "kv_gamma.bin": kc.gamma, "cos_k.bin": kc.cos, "sin_k.bin": kc.sin,
             "index.bin": kc.index, "k_cache.bin": kc.k_cache, "ckv_cache.bin": kc.ckv_cache,
             "k_scale.bin": kc.k_scale, "k_offset.bin": kc.k_offset, "v_scale.bin": kc.v_scale,
             "v_offset.bin": kc.v_offset}
    for name, arr in files.items():
        np.ascontiguousarray(arr).tofile(str(tmp_path / name))
    args = [exe, str(tmp_path), S, H, nq, nkv, d, kc.B, kc.N, kc.S, kc.Dkv, kc.Dv, kc.block_size, kc.block_num]
    r = subprocess.run([str(x) for x in args], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "prologue ok" in r.stdout, r.stdout + r.stderr

    # the row quantiser, bit for bit
    codes = np.fromfile(str(tmp_path / "a_out.bin"), np.uint8).reshape(S, H)
    scale = np.fromfile(str(tmp_path / "a_scale_out.bin"), np.float32)
    c_ref, s_ref = oracle.row_quantize(hidden)
    assert np.array_equal(codes, c_ref) and np.array_equal(scale.view(np.uint32), s_ref.view(np.uint32))
    # the projection with its norms and RoPE, on those codes
    qc.a, qc.a_scale = c_ref, s_ref
    out = np.fromfile(str(tmp_path / "out.bin"), np.uint16).reshape(S, qc.I)
    got = as_f64(torch.from_numpy(out.view(np.int16)).view(torch.bfloat16))
    check_qkv(qc, got, qkv_reference(qc), "prologue from C")
    # the caches
    run = SimpleNamespace(
        k_cache=torch.from_numpy(np.fromfile(str(tmp_path / "k_cache_out.bin"), np.int8).reshape(kc.k_cache.shape)),
        ckv_cache=torch.from_numpy(np.fromfile(str(tmp_path / "ckv_cache_out.bin"), np.int8).reshape(kc.ckv_cache.shape)),
        outputs=False, k_rope=None, c_kv=None,
        err=torch.from_numpy(np.fromfile(str(tmp_path / "err_out.bin"), np.int32)))
    check_kv(kc, run, "KV cache from C")
