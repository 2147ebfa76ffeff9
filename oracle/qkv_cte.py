"""Oracle for the fused QKV projection with across-heads RMSNorm and rotate-half RoPE.

Test infrastructure only (see the package docstring).

Source: AWS Neuron "Kernel reference: qkv_cte -- Wan2.2 additions to the NKI
Library QKV CTE MXFP8 projection".

* Projection: O[S, I] = A[S, H] @ W[H, I] (+ bias), I = (n_q + 2 n_kv) d_head
  (section "Upstream behavior"); A is the row-packed FP8 activation with one
  fp32 dequant scale per row; W is the MX FP8 weight, dequantised while the
  accumulator is read out, then the bias is added (section "Applies to",
  "Pattern").  The MX weight carries a ue8m0 scale per 32-element block along
  H and, optionally, a per-output-channel fp32 scale (section "Interface",
  ``weight_scales``).
* Across-heads RMSNorm (Design 1): per token, one sum of squares over the
  whole Q segment and one over the whole K segment of the un-normalised
  output (1a); inv_rms = rsqrt(sum / width + eps) with width = n_heads*d_head
  for Q and n_kv_heads*d_head for K, tp = 1 (1b); multiply by the
  segment-wide gamma per channel (1c).  V is never normed.
* Rotate-half RoPE (Design 2): lanes (i, i+d/2) of each head pair up;
  out = y*cos + [-y_hi, y_lo]*sin with cos/sin per position, shared by all
  heads.  Wan applies the norm before RoPE, so y already carries inv_rms and
  gamma when it is rotated.
* Single-segment calls (Design 5): num_kv_heads = 0 means I = n_q*d_head and
  the whole projection is normed as Q.

The result is returned unrounded in float64.
"""
from __future__ import annotations

import numpy as np

from .codes import decode_bf16, decode_e4m3, decode_ue8m0

MX_BLOCK = 32


def dequant_activation(a: np.ndarray, a_scale: np.ndarray) -> np.ndarray:
    """A_hat[t, h] = e4m3(a[t, h]) * a_scale[t]."""
    return decode_e4m3(a) * np.asarray(a_scale, dtype=np.float64)[:, None]


def dequant_weight(w: np.ndarray, w_block_exp: np.ndarray,
                   weight_scales: np.ndarray | None = None) -> np.ndarray:
    """W_hat[h, i] = e4m3(w[h, i]) * 2^(e[h // 32, i] - 127) (* weight_scales[i])."""
    H = w.shape[0]
    block_scale = decode_ue8m0(w_block_exp)                    # [H/32, I]
    per_row = np.repeat(block_scale, MX_BLOCK, axis=0)[:H]     # row h takes block h // 32
    w_hat = decode_e4m3(w) * per_row
    if weight_scales is not None:
        w_hat = w_hat * np.asarray(weight_scales, dtype=np.float64)[None, :]
    return w_hat


def project(a, a_scale, w, w_block_exp, weight_scales=None, bias=None) -> np.ndarray:
    """O = A_hat @ W_hat (+ bias): the plain fp64 matrix product."""
    o = dequant_activation(a, a_scale) @ dequant_weight(w, w_block_exp, weight_scales)
    if bias is not None:
        o = o + decode_bf16(bias)[None, :]
    return o


def rms_norm_across_heads(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """One RMS per token over the whole segment, then the segment-wide gamma."""
    width = x.shape[1]
    sum_sq = np.sum(x * x, axis=1)
    inv_rms = 1.0 / np.sqrt(sum_sq / width + eps)
    return x * inv_rms[:, None] * np.asarray(gamma, dtype=np.float64)[None, :]


def rms_norm_per_head(x: np.ndarray, gamma: np.ndarray, eps: float, head_dim: int) -> np.ndarray:
    """The upstream (per-head) qk-norm (qkv_cte page, Design 1: each head's d_head
    slice is normalised by its own RMS), with the per-head [d_head] gamma."""
    T = x.shape[0]
    xh = x.reshape(T, -1, head_dim)
    inv_rms = 1.0 / np.sqrt(np.sum(xh * xh, axis=2) / head_dim + eps)
    y = xh * inv_rms[:, :, None] * np.asarray(gamma, dtype=np.float64)[None, None, :]
    return y.reshape(T, -1)


def rope_rotate_half(y: np.ndarray, cos: np.ndarray, sin: np.ndarray, head_dim: int) -> np.ndarray:
    """Per head: out_lo = y_lo*cos_lo - y_hi*sin_lo; out_hi = y_hi*cos_hi + y_lo*sin_hi."""
    T = y.shape[0]
    half = head_dim // 2
    yh = y.reshape(T, -1, head_dim)
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    lo, hi = yh[..., :half], yh[..., half:]
    out_lo = lo * c[..., :half] - hi * s[..., :half]
    out_hi = hi * c[..., half:] + lo * s[..., half:]
    return np.concatenate([out_lo, out_hi], axis=-1).reshape(T, -1)


def qkv_cte_mx(a, a_scale, w, w_block_exp, *, num_heads: int, num_kv_heads: int, head_dim: int,
               weight_scales=None, bias=None, q_norm=True, k_norm=True,
               q_gamma=None, k_gamma=None, eps: float = 1e-6, fused_rope: bool = False,
               cos=None, sin=None) -> np.ndarray:
    """Full prologue for the given token rows.

    a [T,H] uint8 e4m3 codes; a_scale [T] fp32; w [H,I] uint8 e4m3; w_block_exp
    [H/32,I] uint8 ue8m0; weight_scales [I] fp32 or None; bias [I] bf16 bits or
    None; q_gamma [n_q*d] / k_gamma [n_kv*d] fp32; cos/sin [T,d] fp32 (the rows
    of the tokens in ``a``).  Rows are independent, so any subset of a
    sequence's tokens may be passed.  Returns [T, I] float64.
    q_norm / k_norm: False (none), True or "across" (RMS_NORM_ACROSS_HEADS,
    gamma [n*d]) or "per_head" (the upstream per-head norm, gamma [d]).
    """
    o = project(a, a_scale, w, w_block_exp, weight_scales, bias)
    q_w = num_heads * head_dim
    k_w = num_kv_heads * head_dim
    assert o.shape[1] == q_w + 2 * k_w
    out = o.copy()
    segments = [(0, q_w, q_norm, q_gamma)]
    if num_kv_heads > 0:
        segments.append((q_w, q_w + k_w, k_norm, k_gamma))
    for lo, hi, norm, gamma in segments:
        y = o[:, lo:hi]
        if norm == "per_head":
            y = rms_norm_per_head(y, gamma, eps, head_dim)
        elif norm:
            y = rms_norm_across_heads(y, gamma, eps)
        if fused_rope:
            y = rope_rotate_half(y, cos, sin, head_dim)
        out[:, lo:hi] = y
    return out


def to_nbsd(out: np.ndarray, B: int, S: int, head_dim: int) -> np.ndarray:
    """The NBSd output layout (qkv_cte page, "Interface": output_layout NBSd for the
    cross-attention calls): [B*S, I] -> [I / head_dim, B, S, head_dim], head n being
    columns [n*head_dim, (n+1)*head_dim) in the order Q heads, K heads, V heads."""
    T, I = out.shape
    n = I // head_dim
    res = np.empty((n, B, S, head_dim), dtype=out.dtype)
    for h in range(n):
        res[h] = out[:, h * head_dim:(h + 1) * head_dim].reshape(B, S, head_dim)
    return res
