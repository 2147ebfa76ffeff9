"""Device-side set-up for one operator call: uploads a seeded case (``synth``)
to HBM, allocates outputs and workspace, and invokes the C-ABI through
``native``.  Buffer management only; every step of the computation runs in the
library's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import native, synth


def to_dev(x: np.ndarray | None, device: str = "cuda", half: str = "bf16") -> torch.Tensor | None:
    """numpy -> device tensor; uint16 arrays (16-bit float bit patterns) become
    torch.bfloat16, or torch.float16 with half="fp16"."""
    if x is None:
        return None
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).to(device).view(
            torch.float16 if half == "fp16" else torch.bfloat16)
    return torch.from_numpy(x).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def norm_code(norm) -> int:
    """synth's norm flag (False, True = across heads, "per_head") as an RA_NORM_* value."""
    if norm == "per_head":
        return native.RA_NORM_RMS_PER_HEAD
    return native.RA_NORM_RMS_ACROSS_HEADS if norm else native.RA_NORM_NONE


def qkv_params(c: synth.QKVCase, layout: int = native.RA_LAYOUT_BSD) -> native.QkvCteMxParams:
    """The qkv_cte_mx parameters of a synth.QKVCase (host only)."""
    return native.QkvCteMxParams(
        B=c.B, S=c.S, H=c.H, num_heads=c.num_heads, num_kv_heads=c.num_kv_heads,
        head_dim=c.head_dim, q_norm=norm_code(c.q_norm), k_norm=norm_code(c.k_norm),
        fused_rope=1 if c.fused_rope else 0, norm_eps=c.eps, output_layout=layout)


_KV_QTYPES = {"int8": native.RA_INT8, "e4m3": native.RA_FP8_E4M3, "e5m2": native.RA_FP8_E5M2}


def kv_params(c: synth.KVCase) -> native.KvRmsNormRopeCacheParams:
    """The kv_rms_norm_rope_cache parameters of a synth.KVCase (host only)."""
    qk, qv = c.k_scale is not None, c.v_scale is not None
    half = native.RA_FP16 if c.dtype == "fp16" else native.RA_BF16
    return native.KvRmsNormRopeCacheParams(
        B=c.B, N=c.N, S=c.S, Dkv=c.Dkv, Dv=c.Dv, rope_size=c.rope_size, variant=c.variant,
        cache_mode=synth.CACHE_MODES[c.cache_mode], block_num=c.block_num,
        block_size=c.block_size, kv_dtype=half,
        k_cache_dtype=_KV_QTYPES[c.k_qtype] if qk else half,
        ckv_cache_dtype=_KV_QTYPES[c.v_qtype] if qv else half,
        epsilon=c.eps, is_output_kv=1 if c.is_output_kv else 0,
        rope_s_broadcast=1 if c.rope_broadcast else 0, cache_seq_len=c.cache_seq,
        k_quant_scalar=1 if qk and c.k_scale.shape == (1,) else 0,
        c_kv_quant_scalar=1 if qv and c.v_scale.shape == (1,) else 0)


class QkvRun:
    """Device buffers for one qkv_cte_mx call of a synth.QKVCase."""

    def __init__(self, case: synth.QKVCase, device: str = "cuda", stream=None,
                 layout: int = native.RA_LAYOUT_BSD):
        self.case = case
        c = case
        self.params = qkv_params(c, layout)
        self.a = to_dev(c.a, device)
        self.a_scale = to_dev(c.a_scale, device)
        w = to_dev(c.w, device)
        e = to_dev(c.w_block_exp, device)
        self.w_packed = native.qkv_cte_mx_pack_weight(w, e, stream=stream)
        torch.cuda.synchronize()
        del w, e
        self.weight_scales = to_dev(c.weight_scales, device)
        self.bias = to_dev(c.bias, device)
        self.cos = to_dev(c.cos, device) if c.fused_rope else None
        self.sin = to_dev(c.sin, device) if c.fused_rope else None
        self.q_gamma = to_dev(c.q_gamma, device) if c.q_norm else None
        self.k_gamma = to_dev(c.k_gamma, device) if c.k_norm else None
        shape = (c.T, c.I) if layout == native.RA_LAYOUT_BSD else (c.I // c.head_dim, c.T, c.head_dim)
        self.out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        nws = native.qkv_cte_mx_workspace_bytes(self.params)
        self.workspace = torch.zeros(nws, dtype=torch.uint8, device=device)

    def run(self, stream=None) -> None:
        native.qkv_cte_mx(self.params, self.a, self.a_scale, self.w_packed, self.weight_scales,
                          self.bias, self.cos, self.sin, self.q_gamma, self.k_gamma, self.out,
                          self.workspace, stream)

    def project(self, stream=None) -> None:
        native.qkv_cte_mx_project(self.params, self.a, self.a_scale, self.w_packed,
                                  self.weight_scales, self.bias, self.q_gamma, self.k_gamma, self.out,
                                  self.workspace, stream)

    def norm_rope(self, stream=None) -> None:
        native.qkv_cte_mx_norm_rope(self.params, self.cos, self.sin, self.out, self.workspace, stream)

    def status(self, stream=None) -> int:
        return native.qkv_cte_mx_status(self.workspace, stream)


class KvRun:
    """Device buffers for one kv_rms_norm_rope_cache call of a synth.KVCase."""

    def __init__(self, case: synth.KVCase, device: str = "cuda"):
        self.case = c = case
        qk, qv = c.k_scale is not None, c.v_scale is not None
        self.params = kv_params(c)
        dev = lambda x: to_dev(x, device, c.dtype)
        self.kv = dev(c.kv)
        self.gamma = dev(c.gamma)
        self.cos = dev(c.cos)
        self.sin = dev(c.sin)
        self.index = dev(c.index)
        self.k_cache = dev(c.k_cache)
        self.ckv_cache = dev(c.ckv_cache)
        self.k_scale = dev(c.k_scale)
        self.k_offset = dev(c.k_offset)
        self.v_scale = dev(c.v_scale)
        self.v_offset = dev(c.v_offset)
        self.v = dev(c.v)
        rows = (c.B, c.N, c.S)
        self.outputs = c.is_output_kv and (c.cache_mode != "Norm" or (c.variant == 2 and (qk or qv)))
        fdt = torch.float16 if c.dtype == "fp16" else torch.bfloat16
        self.k_rope = torch.empty(rows + (c.k_width,), dtype=fdt, device=device) if self.outputs else None
        self.c_kv = torch.empty(rows + (c.ckv_width,), dtype=fdt, device=device) if self.outputs else None
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, stream=None) -> None:
        native.kv_rms_norm_rope_cache(
            self.params, self.kv, self.gamma, self.cos, self.sin, self.index, self.k_cache,
            self.ckv_cache, self.k_scale, self.v_scale, self.k_offset, self.v_offset, self.v,
            self.k_rope, self.c_kv, self.err, stream)
