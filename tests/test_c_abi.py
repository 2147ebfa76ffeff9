"""The C ABI from C, on the CPU: include/rope_attention.h compiles as strict C99
(gcc -std=c99 -pedantic -Wall -Wextra -Werror), a C program links against
librope_attention.so and the calls that need no GPU (version, packed-weight and
workspace sizes, host-side rejections with their messages) give the same
answers as through the Python binding."""
import ctypes
import os
import shutil
import subprocess

import pytest

from rope_attention_gb300 import build, native

HERE = os.path.dirname(os.path.abspath(__file__))
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("c_abi") / "abi_host_calls")
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
           os.path.join(HERE, "c", "abi_host_calls.c"), "-o", exe, "-L", libdir, "-lrope_attention",
           f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"C build failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    out = {}
    for ln in r.stdout.splitlines():
        key, _, val = ln.partition(" ")
        out[key] = val
    return out


def test_version_and_sizes_match_the_binding(c_output):
    assert int(c_output["abi"]) == native.ra_abi_version()
    assert int(c_output["packed_status"]) == native.RA_OK
    assert int(c_output["packed_bytes"]) == native.qkv_cte_mx_packed_weight_bytes(5120, 15360)
    p = native.QkvCteMxParams(B=1, S=75600, H=5120, num_heads=40, num_kv_heads=40, head_dim=128,
                              q_norm=native.RA_NORM_RMS_ACROSS_HEADS, k_norm=native.RA_NORM_RMS_ACROSS_HEADS,
                              fused_rope=1, norm_eps=1e-6, output_layout=native.RA_LAYOUT_BSD)
    assert int(c_output["workspace_status"]) == native.RA_OK
    assert int(c_output["workspace_bytes"]) == native.qkv_cte_mx_workspace_bytes(p)


def test_rejections_reach_a_c_caller_with_their_messages(c_output):
    assert int(c_output["bad_h_status"]) == -1  # RA_ERR_INVALID_ARG
    assert "multiple of 128" in c_output["bad_h_message"]
    assert int(c_output["kv_v1_n2_status"]) == -1
    assert "N == 1" in c_output["kv_v1_n2_message"]
    # the same call through the binding's library handle gives the same message
    lib = native.load()
    p = native.QkvCteMxParams(B=1, S=75600, H=5000, num_heads=40, num_kv_heads=40, head_dim=128,
                              q_norm=1, k_norm=1, fused_rope=1, norm_eps=1e-6, output_layout=0)
    n = ctypes.c_size_t()
    assert lib.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == -1
    assert lib.ra_last_error().decode() == c_output["bad_h_message"]


@pytest.mark.parametrize("src", ["example_prologue.c", "prologue_gpu.c"])
def test_call_sequence_example_compiles(src):
    """tests/c/example_prologue.c (the setup / step / status sequence from C with the
    CUDA runtime) and tests/c/prologue_gpu.c (the program the GPU test runs) compile
    as strict C99 here; they need a GPU to run."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = None
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime_api.h")):
            cuda_inc = os.path.join(root, "include")
            break
    if cuda_inc is None:
        pytest.skip("CUDA runtime headers not found")
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
           "-isystem", cuda_inc, "-c", os.path.join(HERE, "c", src), "-o", os.devnull]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
