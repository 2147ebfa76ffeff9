"""The C-ABI boundary, checked on the CPU (no GPU needed, no kernel launched).

* the library loads and exports every function include/rope_attention.h declares;
* every rejection rule of the header returns its status code and a message.
Each rejected call has exactly one violation and fails host-side validation.
Every test here runs with the library's validate-only hook set
(ra_test_validate_only), under which a call that passes its checks returns
before any CUDA runtime call: the placeholder device addresses used here can
never reach a kernel, on this machine or on one with a GPU, whatever the order
of the library's checks.
"""
import ctypes
import os
import re

import pytest

from rope_attention_gb300 import native

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "rope_attention.h")
A16 = 0x10000  # 16-byte aligned placeholder address (never dereferenced)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    from rope_attention_gb300 import build
    build.build()
    lib = native.load()
    lib.ra_test_validate_only(1)
    yield lib
    lib.ra_test_validate_only(0)


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), f"{n} declared in the header but not exported"
    assert sorted(names) == sorted(native.EXPORTS)
    assert native.ra_abi_version() == 9


def test_missing_library_fails_loudly(tmp_path):
    saved = native._LIB
    native._LIB = None
    try:
        with pytest.raises(FileNotFoundError):
            native.load(str(tmp_path / "librope_attention.so"))
    finally:
        native._LIB = saved


def qp(**kw):
    base = dict(B=1, S=256, H=512, num_heads=4, num_kv_heads=4, head_dim=64,
                q_norm=1, k_norm=1, fused_rope=1, norm_eps=1e-6, output_layout=0)
    base.update(kw)
    return native.QkvCteMxParams(**base)


def status_and_msg(L, st):
    return st, L.ra_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(H=100), -1), (dict(H=0), -1), (dict(B=0), -1), (dict(S=0), -1), (dict(num_heads=0), -1),
    (dict(num_kv_heads=-1), -1), (dict(head_dim=24), -1), (dict(q_norm=3), -1),
    (dict(num_kv_heads=0, k_norm=1), -1), (dict(output_layout=2), -1), (dict(output_layout=7), -1),
    (dict(q_norm=2, head_dim=32), -2), (dict(q_norm=3), -1),
    (dict(norm_eps=-1.0), -1), (dict(norm_eps=float("nan")), -1), (dict(fused_rope=2), -1),
])
def test_qkv_params_rejected(L, kw, code):
    n = ctypes.c_size_t()
    st, msg = status_and_msg(L, L.qkv_cte_mx_workspace_bytes(ctypes.byref(qp(**kw)), ctypes.byref(n)))
    assert st == code and msg


def test_workspace_formula(L):
    pad = lambda b: -(-b // 256) * 256
    n = ctypes.c_size_t()
    p = qp(B=1, S=32760, H=5120, num_heads=40, num_kv_heads=40, head_dim=128)
    assert L.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    blocks = (80 * 128) // 128          # 128-column blocks over Q|K (token-major, padded rows)
    assert n.value == 256 + pad(blocks * 32760 * 8) + pad(blocks * 32760)
    p = qp(q_norm=0, k_norm=0, fused_rope=0)
    assert L.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0 and n.value == 256
    p = qp(S=100, q_norm=0, k_norm=0, fused_rope=1)   # RoPE only: exponents for Q|K, no sums
    assert L.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 256 + pad(16 * 100)              # exponent rows padded to 16 bytes
    p = qp(S=100, q_norm=1, k_norm=0, fused_rope=0)   # Q only
    assert L.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 256 + pad(2 * 100 * 8) + pad(16 * 100)


def ws_bytes(L, p):
    n = ctypes.c_size_t()
    assert L.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == 0
    return n.value


def qkv_call(L, p, **over):
    args = dict(a=A16, a_scale=A16, w=A16, ws=None, bias=A16, cos=A16, sin=A16, qg=A16, kg=A16,
                out=A16, work=A16, nwork=ws_bytes(L, p))
    args.update(over)
    return L.qkv_cte_mx(ctypes.byref(p), args["a"], args["a_scale"], args["w"], args["ws"], args["bias"],
                        args["cos"], args["sin"], args["qg"], args["kg"], args["out"], args["work"],
                        args["nwork"], None)


@pytest.mark.parametrize("over,code", [
    (dict(cos=None), -1), (dict(sin=None), -1), (dict(qg=None), -1), (dict(kg=None), -1),
    (dict(a=None), -1), (dict(out=None), -1), (dict(work=None), -1), (dict(w=None), -1),
    (dict(a=A16 + 1), -3), (dict(out=A16 + 8), -3), (dict(bias=A16 + 2), -3), (dict(cos=A16 + 4), -3),
    (dict(work=A16 + 4), -3), (dict(nwork=16), -4),
])
def test_qkv_call_rejected(L, over, code):
    if "nwork" in over:
        assert ws_bytes(L, qp()) > over["nwork"]   # placeholders: the call must be refused
    st, msg = status_and_msg(L, qkv_call(L, qp(), **over))
    assert st == code and msg


def test_project_and_norm_rejections(L):
    p = qp()
    assert ws_bytes(L, p) > 8   # the 8-byte workspace below is always refused
    st = L.qkv_cte_mx_project(ctypes.byref(p), A16, A16, A16, None, None, A16, A16, A16, A16, 8, None)
    assert st == -4
    st = L.qkv_cte_mx_project(ctypes.byref(p), A16, A16, A16, None, None, None, A16, A16, A16,
                              ws_bytes(L, p), None)
    assert st == -1                                          # q_norm needs q_gamma
    ph = qp(q_norm=2, k_norm=2, head_dim=64)
    st = L.qkv_cte_mx_project(ctypes.byref(ph), A16, A16, A16, None, None, A16, None, A16, A16,
                              ws_bytes(L, ph), None)
    assert st == -1 and b"k_gamma" in L.ra_last_error()     # the per-head K norm needs its gamma
    st = L.qkv_cte_mx_norm_rope(ctypes.byref(p), None, A16, A16, A16, ws_bytes(L, p), None)
    assert st == -1                                          # fused_rope needs cos/sin
    assert L.qkv_cte_mx_status(None, None, None) == -1           # device_status is required
    assert L.kv_rms_norm_rope_cache_status(None, None) == -1    # device_status is required


def test_pack_weight_rejections(L):
    n = ctypes.c_size_t()
    assert L.qkv_cte_mx_packed_weight_bytes(100, 384, ctypes.byref(n)) == -1
    assert L.qkv_cte_mx_packed_weight_bytes(256, 100, ctypes.byref(n)) == -1
    assert L.qkv_cte_mx_packed_weight_bytes(256, 384, ctypes.byref(n)) == 0
    need = n.value
    assert need >= 256 * 384
    assert L.qkv_cte_mx_pack_weight(A16, A16, 256, 384, A16, need - 1, None) == -4
    assert L.qkv_cte_mx_pack_weight(A16, A16, 256, 384, A16 + 4, need, None) == -3
    assert L.qkv_cte_mx_pack_weight(None, A16, 256, 384, A16, need, None) == -1


def kp(**kw):
    base = dict(B=2, N=1, S=64, Dkv=576, Dv=512, rope_size=64, variant=1, cache_mode=2,
                block_num=4, block_size=32, kv_dtype=0, k_cache_dtype=0, ckv_cache_dtype=0,
                epsilon=1e-5, is_output_kv=0)
    base.update(kw)
    return native.KvRmsNormRopeCacheParams(**base)


def kv_call(L, p, **over):
    args = dict(kv=A16, gamma=A16, cos=A16, sin=A16, index=A16, kc=A16, cc=A16, ks=None, vs=None,
                ko=None, vo=None, v=None, kr=None, ckv=None, err=None)
    args.update(over)
    return L.kv_rms_norm_rope_cache(ctypes.byref(p), args["kv"], args["gamma"], args["cos"], args["sin"],
                                    args["index"], args["kc"], args["cc"], args["ks"], args["vs"],
                                    args["ko"], args["vo"], args["v"], args["kr"], args["ckv"],
                                    args["err"], None)


@pytest.mark.parametrize("pkw,over,code", [
    (dict(N=2), {}, -1),                                        # V1 needs N == 1
    (dict(variant=2, N=3, Dkv=192, Dv=128), dict(v=A16), -1),   # V2 needs N in {1,2,4,8}
    (dict(variant=2, N=2, Dkv=192, Dv=128), {}, -1),            # V2 needs v_optional
    ({}, dict(v=A16), -1),                                      # V1 takes no v_optional
    (dict(variant=3), {}, -1),
    (dict(B=0), {}, -1), (dict(S=0), {}, -1),                   # no empty tensors
    (dict(rope_size=6, Dv=570), {}, -1),                        # rope width (multiple of 8 here)
    (dict(Dv=500), {}, -1),                                     # V1: Dv = Dkv - rope
    ({}, dict(ko=A16), -1),                                     # offset without scale
    ({}, dict(vs=A16), -1),                                     # quant with a bf16 cache
    (dict(k_cache_dtype=2), {}, -1),                            # int8 cache without scale
    (dict(k_cache_dtype=2, ckv_cache_dtype=2, block_size=48), dict(ks=A16, vs=A16), -1),
    (dict(block_size=24), {}, -1),                              # bf16 caches need %16
    (dict(block_size=1), {}, -1),
    (dict(cache_mode=0), {}, -1),                               # Norm needs cache_seq_len >= S
    (dict(cache_mode=0, cache_seq_len=64, k_cache_dtype=2), dict(ks=A16), -1),  # V1 Norm: no quant
    (dict(cache_mode=3), {}, -2), (dict(cache_mode=5), {}, -2),  # FRACTAL_NZ modes not built
    (dict(cache_mode=6), {}, -1),                               # unknown mode
    (dict(kv_dtype=3, k_cache_dtype=3, ckv_cache_dtype=3), {}, -1),  # fp32 kv
    (dict(k_cache_dtype=3), dict(ks=A16), -1),                  # fp32 is not a quantised cache type
    (dict(k_cache_dtype=4, ckv_cache_dtype=5, block_size=48), dict(ks=A16, vs=A16), -1),  # 1-byte: %32
    (dict(rope_s_broadcast=2), {}, -1),
    (dict(k_quant_scalar=2, k_cache_dtype=2), dict(ks=A16), -1),   # flag is 0 or 1
    (dict(k_quant_scalar=1), {}, -1),                           # [1] flag without its scale
    (dict(variant=2, N=2, Dkv=192, Dv=128, k_cache_dtype=2, k_quant_scalar=1),
     dict(v=A16, ks=A16), -1),                                  # V2 parameters are [N, D]
    (dict(is_output_kv=1), {}, -1),                             # needs k_rope / c_kv
    (dict(epsilon=-1.0), {}, -1),
    ({}, dict(kv=A16 + 2), -3), ({}, dict(index=A16 + 4), -3), ({}, dict(kc=A16 + 8), -3),
    ({}, dict(kv=None), -1), ({}, dict(index=None), -1),
])
def test_kv_rejected(L, pkw, over, code):
    st, msg = status_and_msg(L, kv_call(L, kp(**pkw), **over))
    assert st == code and msg, (st, msg)


# ---------------------------------------------------------------- row quantiser
@pytest.mark.parametrize("what,args,status,msg", [
    ("null x", (None, 4, 64, A16, A16), -1, "required"),
    ("null codes", (A16, 4, 64, None, A16), -1, "required"),
    ("null scale", (A16, 4, 64, A16, None), -1, "required"),
    ("no rows", (A16, 0, 64, A16, A16), -1, "multiple of 8"),
    ("H not a multiple of 8", (A16, 4, 60, A16, A16), -1, "multiple of 8"),
    ("x misaligned", (A16 + 8, 4, 64, A16, A16), -3, "x must be"),
    ("codes misaligned", (A16, 4, 64, A16 + 4, A16), -3, "aligned"),
    ("scale misaligned", (A16, 4, 64, A16, A16 + 2), -3, "aligned"),
])
def test_row_quantize_rejections(L, what, args, status, msg):
    x, T, H, codes, scale = args
    st = L.row_quantize_e4m3(x, T, H, codes, scale, None)
    assert st == status, what
    assert msg in L.ra_last_error().decode(), what


@pytest.mark.parametrize("what,args,status", [
    ("null packed", (A16, 4, 64, None), -1),
    ("H not a multiple of 8", (A16, 4, 12, A16), -1),
    ("packed misaligned", (A16, 4, 64, A16 + 2), -3),
])
def test_row_quantize_packed_rejections(L, what, args, status):
    assert L.row_quantize_e4m3_packed(*args, None) == status, what


# ---------------------------------------------------------------- the validate-only hook
def valid_calls(L):
    """One call per launching entry point, each passing every host check."""
    p = qp()
    n = ws_bytes(L, p)
    k = kp(variant=2, N=2, Dkv=192, Dv=128, k_cache_dtype=2, ckv_cache_dtype=2)
    return {
        "qkv_cte_mx": lambda: qkv_call(L, p),
        "qkv_cte_mx_project": lambda: L.qkv_cte_mx_project(ctypes.byref(p), A16, A16, A16, None, None, A16, A16,
                                                           A16, A16, n, None),
        "qkv_cte_mx_norm_rope": lambda: L.qkv_cte_mx_norm_rope(ctypes.byref(p), A16, A16, A16, A16, n, None),
        "qkv_cte_mx_noalloc": lambda: L.qkv_cte_mx_noalloc(ctypes.byref(p), A16, A16, A16, None, A16, A16, A16,
                                                           A16, A16, A16, None),
        "qkv_cte_mx_pack_weight": lambda: L.qkv_cte_mx_pack_weight(A16, A16, 256, 384, A16, 1 << 30, None),
        "kv_rms_norm_rope_cache": lambda: kv_call(L, k, v=A16, ks=A16, vs=A16),
        "row_quantize_e4m3": lambda: L.row_quantize_e4m3(A16, 4, 64, A16, A16, None),
        "row_quantize_e4m3_packed": lambda: L.row_quantize_e4m3_packed(A16, 4, 64, A16, None),
    }


def test_validate_only_returns_before_any_cuda_call(L):
    """With the hook set (as for every test in this file), a call that passes its host
    checks returns RA_OK without touching CUDA, and the status readers report 0."""
    for name, call in valid_calls(L).items():
        assert call() == 0, (name, L.ra_last_error())
    v = ctypes.c_int32(7)
    assert L.qkv_cte_mx_status(A16, None, ctypes.byref(v)) == 0 and v.value == 0
    v = ctypes.c_int32(7)
    assert L.qkv_cte_mx_status(None, None, ctypes.byref(v)) == 0 and v.value == 0
    v = ctypes.c_int32(7)
    assert L.kv_rms_norm_rope_cache_status(None, ctypes.byref(v)) == 0 and v.value == 0


def test_validate_only_is_what_stops_the_launch(L):
    """Without the hook the same valid calls go on to the CUDA runtime, which on a
    machine without a GPU fails (RA_ERR_CUDA): so it is the hook, not a check,
    that keeps the placeholder addresses away from the device.  Runs only where no
    GPU is visible, since these calls would otherwise launch on those addresses."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on placeholder addresses with a GPU present")
    calls = valid_calls(L)
    L.ra_test_validate_only(0)
    try:
        for name, call in calls.items():
            assert call() == -5, (name, L.ra_last_error())  # RA_ERR_CUDA: no device here
    finally:
        L.ra_test_validate_only(1)
