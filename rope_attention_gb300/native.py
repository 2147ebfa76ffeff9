"""ctypes binding of librope_attention.so (include/rope_attention.h).

Argument marshalling only: every function here checks tensor placement,
dtype, contiguity and size, turns tensors into raw pointers and calls the C
entry point of the same name on the current CUDA stream.  The C ABI takes bare
pointers, so it cannot see how large a buffer is; the binding refuses a tensor
smaller than the extent the call reads or writes through it (``qkv_extents``,
``kv_extents``) before anything reaches the device.  All arithmetic happens in
the library's CUDA kernels; there is no CPU fallback.  ``load()`` raises if
the library has not been built (``python -m rope_attention_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

RA_OK = 0
STATUS_NAMES = {0: "RA_OK", -1: "RA_ERR_INVALID_ARG", -2: "RA_ERR_UNSUPPORTED",
                -3: "RA_ERR_ALIGNMENT", -4: "RA_ERR_WORKSPACE", -5: "RA_ERR_CUDA",
                -6: "RA_ERR_TIMEOUT", -7: "RA_ERR_INDEX"}
RA_BF16, RA_FP16, RA_INT8, RA_FP32, RA_FP8_E4M3, RA_FP8_E5M2 = 0, 1, 2, 3, 4, 5
RA_NORM_NONE, RA_NORM_RMS_ACROSS_HEADS, RA_NORM_RMS_PER_HEAD = 0, 1, 2
RA_LAYOUT_BSD, RA_LAYOUT_NBSD = 0, 1
RA_CACHE_NORM, RA_CACHE_PA, RA_CACHE_PA_BNSD, RA_CACHE_PA_NZ, RA_CACHE_PA_BLK_BNSD, RA_CACHE_PA_BLK_NZ = \
    0, 1, 2, 3, 4, 5

EXPORTS = ["ra_last_error", "ra_abi_version", "ra_set_wait_timeout_ns", "ra_test_stall_next_projection",
           "qkv_cte_mx_packed_weight_bytes", "qkv_cte_mx_pack_weight", "qkv_cte_mx_workspace_bytes",
           "qkv_cte_mx", "qkv_cte_mx_project", "qkv_cte_mx_norm_rope", "qkv_cte_mx_status",
           "qkv_cte_mx_noalloc", "kv_rms_norm_rope_cache", "kv_rms_norm_rope_cache_status",
           "ra_test_stall_next_kv_cache", "ra_test_stall_next_norm_rope", "row_quantize_e4m3",
           "row_quantize_e4m3_packed", "ra_test_validate_only"]


class RAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class QkvCteMxParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("S", ctypes.c_int64), ("H", ctypes.c_int64),
                ("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("q_norm", ctypes.c_int32), ("k_norm", ctypes.c_int32),
                ("fused_rope", ctypes.c_int32), ("norm_eps", ctypes.c_float),
                ("output_layout", ctypes.c_int32)]


class KvRmsNormRopeCacheParams(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("N", ctypes.c_int64), ("S", ctypes.c_int64),
                ("Dkv", ctypes.c_int64), ("Dv", ctypes.c_int64), ("rope_size", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("cache_mode", ctypes.c_int32),
                ("block_num", ctypes.c_int64), ("block_size", ctypes.c_int64),
                ("kv_dtype", ctypes.c_int32), ("k_cache_dtype", ctypes.c_int32),
                ("ckv_cache_dtype", ctypes.c_int32), ("epsilon", ctypes.c_float),
                ("is_output_kv", ctypes.c_int32), ("rope_s_broadcast", ctypes.c_int32),
                ("cache_seq_len", ctypes.c_int64), ("k_quant_scalar", ctypes.c_int32),
                ("c_kv_quant_scalar", ctypes.c_int32)]


_LIB = None
P = ctypes.c_void_p


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (once).  Raises FileNotFoundError if it is not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with `python -m rope_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "ra_last_error": (ctypes.c_char_p, []),
        "ra_abi_version": (i32, []),
        "ra_set_wait_timeout_ns": (None, [i64]),
        "ra_test_stall_next_projection": (None, []),
        "qkv_cte_mx_packed_weight_bytes": (i32, [i64, i64, ctypes.POINTER(sz)]),
        "qkv_cte_mx_pack_weight": (i32, [P, P, i64, i64, P, sz, P]),
        "qkv_cte_mx_workspace_bytes": (i32, [ctypes.POINTER(QkvCteMxParams), ctypes.POINTER(sz)]),
        "qkv_cte_mx": (i32, [ctypes.POINTER(QkvCteMxParams), P, P, P, P, P, P, P, P, P, P, P, sz, P]),
        "qkv_cte_mx_project": (i32, [ctypes.POINTER(QkvCteMxParams), P, P, P, P, P, P, P, P, P, sz, P]),
        "qkv_cte_mx_norm_rope": (i32, [ctypes.POINTER(QkvCteMxParams), P, P, P, P, sz, P]),
        "qkv_cte_mx_status": (i32, [P, P, ctypes.POINTER(i32)]),
        "qkv_cte_mx_noalloc": (i32, [ctypes.POINTER(QkvCteMxParams), P, P, P, P, P, P, P, P, P, P, P]),
        "kv_rms_norm_rope_cache": (i32, [ctypes.POINTER(KvRmsNormRopeCacheParams), P, P, P, P, P,
                                         P, P, P, P, P, P, P, P, P, P, P]),
        "kv_rms_norm_rope_cache_status": (i32, [P, ctypes.POINTER(i32)]),
        "ra_test_stall_next_kv_cache": (None, []),
        "ra_test_stall_next_norm_rope": (None, []),
        "row_quantize_e4m3": (i32, [P, i64, i64, P, P, P]),
        "row_quantize_e4m3_packed": (i32, [P, i64, i64, P, P]),
        "ra_test_validate_only": (None, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != RA_OK:
        raise RAError(status, load().ra_last_error().decode())


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _need(t: torch.Tensor | None, nbytes: int, name: str) -> None:
    """Raise if ``t`` spans fewer bytes than the call reads or writes through it."""
    if t is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: the call needs {nbytes} bytes, the tensor holds "
                         f"{t.numel() * t.element_size()}")


def _need_all(ext: dict[str, int], **tensors) -> None:
    for name, t in tensors.items():
        _need(t, ext[name], name)


def qkv_extents(p: QkvCteMxParams) -> dict[str, int]:
    """Bytes that each tensor argument of the qkv_cte_mx calls spans, from the
    call's parameters (header comments of qkv_cte_mx).  Optional arguments get
    the extent they have when given; cos/sin and the gammas count only when
    fused_rope / the segment's norm are on (otherwise the call ignores them).
    Parameters the library rejects give meaningless extents; the library's own
    validation answers for those."""
    B, S, H = max(p.B, 0), max(p.S, 0), max(p.H, 0)
    T, d = B * S, max(p.head_dim, 0)
    nq, nk = max(p.num_heads, 0), max(p.num_kv_heads, 0)
    I = (nq + 2 * nk) * d

    def gamma(norm: int, n: int) -> int:
        return {RA_NORM_RMS_ACROSS_HEADS: n * d * 4, RA_NORM_RMS_PER_HEAD: d * 4}.get(norm, 0)

    rope = T * d * 4 if p.fused_rope == 1 else 0
    return {"a": T * H, "a_scale": T * 4, "weight_scales": I * 4, "bias": I * 2,
            "cos_cache": rope, "sin_cache": rope, "q_gamma": gamma(p.q_norm, nq),
            "k_gamma": gamma(p.k_norm, nk) if nk > 0 else 0, "out": T * I * 2}


_CACHE_BYTES = {RA_BF16: 2, RA_FP16: 2, RA_INT8: 1, RA_FP8_E4M3: 1, RA_FP8_E5M2: 1}


def kv_extents(p: KvRmsNormRopeCacheParams) -> dict[str, int]:
    """Bytes that each tensor argument of kv_rms_norm_rope_cache spans, from the
    call's parameters (header comments of kv_rms_norm_rope_cache and RA_CACHE_*):
    caches [block_num, N, block_size, D] / [block_num, block_size, N, D] in the
    paged modes and [B, N, cache_seq_len, D] in NORM mode; index [B*S], or
    [B * ceil(S / block_size)] in PA_BLK_BNSD; quantisation parameters [D] ([1]
    with the scalar flag) in V1 and [N, D] in V2.  Parameters the library rejects
    give meaningless extents; the library's own validation answers for those."""
    B, N, S = max(p.B, 0), max(p.N, 0), max(p.S, 0)
    Dkv, Dv, R = max(p.Dkv, 0), max(p.Dv, 0), max(p.rope_size, 0)
    v1 = p.variant == 1
    rms = max(Dkv - R, 0) if v1 else Dkv
    kw, cw = (R, rms) if v1 else (Dkv, Dv)
    rows = B * N * S
    bs = max(p.block_size, 1)
    if p.cache_mode == RA_CACHE_NORM:
        slots, n_index = B * max(p.cache_seq_len, 0), B * S
    elif p.cache_mode == RA_CACHE_PA_BLK_BNSD:
        slots, n_index = max(p.block_num, 0) * bs, B * (-(-S // bs))
    else:
        slots, n_index = max(p.block_num, 0) * bs, B * S
    qk = (1 if p.k_quant_scalar else kw) if v1 else N * kw
    qv = (1 if p.c_kv_quant_scalar else cw) if v1 else N * cw
    rope_rows = B * N * (1 if p.rope_s_broadcast else S)
    # k_rope / c_kv are written (and otherwise ignored) per the combination table:
    # with is_output_kv, and in NORM mode only for V2 with a quantised cache
    quant = p.k_cache_dtype not in (RA_BF16, RA_FP16) or p.ckv_cache_dtype not in (RA_BF16, RA_FP16)
    outputs = bool(p.is_output_kv) and (p.cache_mode != RA_CACHE_NORM or (not v1 and quant))
    return {"kv": rows * Dkv * 2, "gamma": rms * 2, "cos": rope_rows * R * 2, "sin": rope_rows * R * 2,
            "index": n_index * 8,
            "k_cache": slots * N * kw * _CACHE_BYTES.get(p.k_cache_dtype, 1),
            "ckv_cache": slots * N * cw * _CACHE_BYTES.get(p.ckv_cache_dtype, 1),
            "k_rope_scale": qk * 4, "k_rope_offset": qk * 4, "c_kv_scale": qv * 4, "c_kv_offset": qv * 4,
            "v_optional": rows * Dv * 2, "k_rope": rows * kw * 2 if outputs else 0,
            "c_kv": rows * cw * 2 if outputs else 0,
            "dev_error_count": 4}


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bits16(t: torch.Tensor | None) -> torch.Tensor | None:
    """bf16 / fp16 tensors are passed as their 16-bit patterns."""
    if t is None:
        return None
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.float16) else t


def ra_abi_version() -> int:
    return int(load().ra_abi_version())


def ra_set_wait_timeout_ns(ns: int) -> None:
    load().ra_set_wait_timeout_ns(int(ns))


def ra_test_validate_only(on: bool) -> None:
    """Test hook: while on, every call returns right after its host checks (no CUDA call)."""
    load().ra_test_validate_only(1 if on else 0)


def ra_test_stall_next_projection() -> None:
    """Test hook: the next projection launch issues no loads, so its waits time out."""
    load().ra_test_stall_next_projection()


def ra_test_stall_next_norm_rope() -> None:
    """Test hook: the next pipelined norm/RoPE launch issues no copies, so its waits time out."""
    load().ra_test_stall_next_norm_rope()


def ra_test_stall_next_kv_cache() -> None:
    """Test hook: the next pipelined KV cache launch issues no copies, so its waits time out."""
    load().ra_test_stall_next_kv_cache()


# ---------------------------------------------------------------- qkv_cte_mx
def qkv_cte_mx_packed_weight_bytes(H: int, I: int) -> int:
    n = ctypes.c_size_t()
    _check(load().qkv_cte_mx_packed_weight_bytes(H, I, ctypes.byref(n)))
    return n.value


def qkv_cte_mx_pack_weight(w: torch.Tensor, w_block_exp: torch.Tensor, packed: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """w [H, I] uint8 e4m3 codes, w_block_exp [H/32, I] uint8; returns the packed uint8 buffer."""
    H, I = w.shape
    nbytes = qkv_cte_mx_packed_weight_bytes(H, I)
    _need(w_block_exp, (H // 32) * I, "w_block_exp")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    _check(load().qkv_cte_mx_pack_weight(_ptr(w, torch.uint8, "w"), _ptr(w_block_exp, torch.uint8, "w_block_exp"),
                                         H, I, _ptr(packed, torch.uint8, "packed"), packed.numel(),
                                         _stream(stream)))
    return packed


def qkv_cte_mx_workspace_bytes(params: QkvCteMxParams) -> int:
    n = ctypes.c_size_t()
    _check(load().qkv_cte_mx_workspace_bytes(ctypes.byref(params), ctypes.byref(n)))
    return n.value


def _need_w_packed(params, w_packed) -> None:
    I = (max(params.num_heads, 0) + 2 * max(params.num_kv_heads, 0)) * max(params.head_dim, 0)
    try:
        nbytes = qkv_cte_mx_packed_weight_bytes(params.H, I)
    except RAError:
        return  # shapes the library rejects: the call itself reports them
    _need(w_packed, nbytes, "w_packed")


def qkv_cte_mx(params, a, a_scale, w_packed, weight_scales, bias, cos_cache, sin_cache, q_gamma,
               k_gamma, out, workspace, stream=None) -> None:
    _need_all(qkv_extents(params), a=a, a_scale=a_scale, weight_scales=weight_scales, bias=bias,
              cos_cache=cos_cache, sin_cache=sin_cache, q_gamma=q_gamma, k_gamma=k_gamma, out=out)
    _need_w_packed(params, w_packed)
    _check(load().qkv_cte_mx(
        ctypes.byref(params), _ptr(a, torch.uint8, "a"), _ptr(a_scale, torch.float32, "a_scale"),
        _ptr(w_packed, torch.uint8, "w_packed"), _ptr(weight_scales, torch.float32, "weight_scales"),
        _ptr(_bits16(bias), None, "bias"), _ptr(cos_cache, torch.float32, "cos_cache"),
        _ptr(sin_cache, torch.float32, "sin_cache"), _ptr(q_gamma, torch.float32, "q_gamma"),
        _ptr(k_gamma, torch.float32, "k_gamma"), _ptr(_bits16(out), None, "out"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def qkv_cte_mx_project(params, a, a_scale, w_packed, weight_scales, bias, q_gamma, k_gamma, out, workspace,
                       stream=None) -> None:
    _need_all(qkv_extents(params), a=a, a_scale=a_scale, weight_scales=weight_scales, bias=bias,
              q_gamma=q_gamma, k_gamma=k_gamma, out=out)
    _need_w_packed(params, w_packed)
    _check(load().qkv_cte_mx_project(
        ctypes.byref(params), _ptr(a, torch.uint8, "a"), _ptr(a_scale, torch.float32, "a_scale"),
        _ptr(w_packed, torch.uint8, "w_packed"), _ptr(weight_scales, torch.float32, "weight_scales"),
        _ptr(_bits16(bias), None, "bias"), _ptr(q_gamma, torch.float32, "q_gamma"),
        _ptr(k_gamma, torch.float32, "k_gamma"), _ptr(_bits16(out), None, "out"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def qkv_cte_mx_norm_rope(params, cos_cache, sin_cache, out, workspace, stream=None) -> None:
    _need_all(qkv_extents(params), cos_cache=cos_cache, sin_cache=sin_cache, out=out)
    _check(load().qkv_cte_mx_norm_rope(
        ctypes.byref(params), _ptr(cos_cache, torch.float32, "cos_cache"),
        _ptr(sin_cache, torch.float32, "sin_cache"), _ptr(_bits16(out), None, "out"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def qkv_cte_mx_noalloc(params, a, a_scale, w_packed, weight_scales, bias, cos_cache, sin_cache,
                       q_gamma, k_gamma, out, stream=None) -> None:
    """qkv_cte_mx with the library's static device workspace (no allocation anywhere)."""
    _need_all(qkv_extents(params), a=a, a_scale=a_scale, weight_scales=weight_scales, bias=bias,
              cos_cache=cos_cache, sin_cache=sin_cache, q_gamma=q_gamma, k_gamma=k_gamma, out=out)
    _need_w_packed(params, w_packed)
    _check(load().qkv_cte_mx_noalloc(
        ctypes.byref(params), _ptr(a, torch.uint8, "a"), _ptr(a_scale, torch.float32, "a_scale"),
        _ptr(w_packed, torch.uint8, "w_packed"), _ptr(weight_scales, torch.float32, "weight_scales"),
        _ptr(_bits16(bias), None, "bias"), _ptr(cos_cache, torch.float32, "cos_cache"),
        _ptr(sin_cache, torch.float32, "sin_cache"), _ptr(q_gamma, torch.float32, "q_gamma"),
        _ptr(k_gamma, torch.float32, "k_gamma"), _ptr(_bits16(out), None, "out"), _stream(stream)))


def qkv_cte_mx_status(workspace: torch.Tensor | None, stream=None) -> int:
    """Synchronises the stream; returns the device status word (0 = fine) and clears it.
    workspace None: the static workspace of qkv_cte_mx_noalloc on the current device."""
    v = ctypes.c_int32()
    st = load().qkv_cte_mx_status(_ptr(workspace, torch.uint8, "workspace"), _stream(stream), ctypes.byref(v))
    if st not in (RA_OK, -6):
        _check(st)
    return v.value


# ---------------------------------------------------------------- kv_rms_norm_rope_cache
def kv_rms_norm_rope_cache_status(stream=None) -> int:
    """Synchronises the stream; returns the KV status word (0 = fine) and clears it."""
    v = ctypes.c_int32()
    st = load().kv_rms_norm_rope_cache_status(_stream(stream), ctypes.byref(v))
    if st not in (RA_OK, -6):
        _check(st)
    return v.value


def kv_rms_norm_rope_cache(params, kv, gamma, cos, sin, index, k_cache, ckv_cache, k_rope_scale=None,
                           c_kv_scale=None, k_rope_offset=None, c_kv_offset=None, v_optional=None,
                           k_rope=None, c_kv=None, dev_error_count=None, stream=None) -> None:
    _need_all(kv_extents(params), kv=kv, gamma=gamma, cos=cos, sin=sin, index=index, k_cache=k_cache,
              ckv_cache=ckv_cache, k_rope_scale=k_rope_scale, c_kv_scale=c_kv_scale,
              k_rope_offset=k_rope_offset, c_kv_offset=c_kv_offset, v_optional=v_optional,
              k_rope=k_rope, c_kv=c_kv, dev_error_count=dev_error_count)
    _check(load().kv_rms_norm_rope_cache(
        ctypes.byref(params), _ptr(_bits16(kv), None, "kv"), _ptr(_bits16(gamma), None, "gamma"),
        _ptr(_bits16(cos), None, "cos"), _ptr(_bits16(sin), None, "sin"), _ptr(index, torch.int64, "index"),
        _ptr(_bits16(k_cache), None, "k_cache"), _ptr(_bits16(ckv_cache), None, "ckv_cache"),
        _ptr(k_rope_scale, torch.float32, "k_rope_scale"), _ptr(c_kv_scale, torch.float32, "c_kv_scale"),
        _ptr(k_rope_offset, torch.float32, "k_rope_offset"), _ptr(c_kv_offset, torch.float32, "c_kv_offset"),
        _ptr(_bits16(v_optional), None, "v_optional"), _ptr(_bits16(k_rope), None, "k_rope"),
        _ptr(_bits16(c_kv), None, "c_kv"), _ptr(dev_error_count, torch.int32, "dev_error_count"),
        _stream(stream)))


# ---------------------------------------------------------------- row quantisation
def row_quantize_e4m3(x: torch.Tensor, codes: torch.Tensor, scale: torch.Tensor, stream=None) -> None:
    """x [T, H] bf16 -> codes [T, H] uint8 (E4M3) and scale [T] float32, on the device."""
    T, H = x.shape
    _need(codes, T * H, "codes")
    _need(scale, T * 4, "scale")
    _check(load().row_quantize_e4m3(_ptr(x, torch.bfloat16, "x"), T, H, _ptr(codes, torch.uint8, "codes"),
                                    _ptr(scale, torch.float32, "scale"), _stream(stream)))


def row_quantize_e4m3_packed(x: torch.Tensor, packed: torch.Tensor, stream=None) -> None:
    """x [T, H] bf16 -> packed [T, H + 4] uint8 (codes, then the fp32 scale's bytes)."""
    T, H = x.shape
    _need(packed, T * (H + 4), "packed")
    _check(load().row_quantize_e4m3_packed(_ptr(x, torch.bfloat16, "x"), T, H,
                                           _ptr(packed, torch.uint8, "packed"), _stream(stream)))
