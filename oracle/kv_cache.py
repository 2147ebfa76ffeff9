"""Oracle for KvRmsNormRopeCache.  Test infrastructure only (see the package docstring).

Source: CANN ops-transformer "KvRmsNormRopeCache" (posembedding), section
"计算公式" (formulas), items (1)-(5), the parameter table, and the
cache/index constraint table.

For kv [B, N, S, Dkv] (and v_optional [B, N, S, Dv] in the separate-kv mode):

(1) RmsNorm: x = kv[..., :rms_size];  y = x / sqrt(mean(x^2) + eps) * gamma.
    V1 (combined kv, no v_optional): rms_size = Dv = Dkv - rope_size.
    V2 (separate kv, v_optional given): rms_size = Dkv.
(2) interleaved RoPE on x_r = kv[..., Dv:] (V1) or y[..., :rope_size] (V2):
    x1 = x_r[..., 0::2], x2 = x_r[..., 1::2],
    y_rope = cat(x1, x2) * cos + cat(-x2, x1) * sin;
    rope_out = y_rope (V1) or cat(y_rope, y[..., rope_size:]) (V2).
(3) Quant (each of k and v independently): x*scale, then +offset, then
    round().clamp(-128, 127) when a scale is given; otherwise x itself.
    ``round`` is read as round-half-to-even (torch semantics, as the formulas
    are written in torch notation).
(4) Scatter: slot p = index[b*S + s]; k_cache[p] <- Quant(rope_out)[b, n, s],
    ckv_cache[p] <- Quant(y)[b, n, s] (V1) or Quant(v)[b, n, s] (V2).  p = -1
    is skipped.  Paged layouts: PA = [block_num, block_size, N, D],
    PA_BNSD = [block_num, N, block_size, D]; p maps to block p // block_size,
    offset p % block_size.
(5) When is_output_kv: k_rope = rope_out and c_kv = y (V1) or v (V2).

Quant scales/offsets are per channel: shape [D] for V1, [N, D] for V2.
Values are computed in float64; bf16 caches receive the unrounded value (the
comparison applies the bf16 tolerance), int8 caches receive the int code, and
the pre-rounding value of every code is returned for the tie rule.
"""
from __future__ import annotations

import numpy as np

from .codes import decode_bf16


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    n = x.shape[-1]
    rms = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) / n + eps)
    return x / rms * gamma


def interleave_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    x1 = x[..., 0::2]
    x2 = x[..., 1::2]
    part1 = np.concatenate([x1, x2], axis=-1)
    part2 = np.concatenate([-x2, x1], axis=-1)
    return part1 * cos + part2 * sin


def quantize(x: np.ndarray, scale, offset, n_axis_param: bool):
    """Returns (value, pre_round).  ``value`` is int64 codes when a scale is given."""
    if scale is None:
        return x, None
    sc = np.asarray(scale, dtype=np.float64)
    if n_axis_param:  # [N, D] broadcast over [B, N, S, D]
        sc = sc[None, :, None, :]
    v = x * sc
    if offset is not None:
        of = np.asarray(offset, dtype=np.float64)
        if n_axis_param:
            of = of[None, :, None, :]
        v = v + of
    return np.clip(np.rint(v), -128, 127).astype(np.int64), v


def kv_rms_norm_rope_cache(kv, gamma, cos, sin, index, k_cache, ckv_cache, *, variant: int,
                           rope_size: int, block_size: int, cache_mode: str = "PA_BNSD",
                           epsilon: float = 1e-5, k_scale=None, k_offset=None, v_scale=None,
                           v_offset=None, v=None, is_output_kv: bool = False) -> dict:
    """Run the operator on host arrays.

    kv, gamma, cos, sin, v: bf16 bit patterns (uint16).  index: int64 [B*S].
    k_cache / ckv_cache: the caches before the call (uint16 bf16 bits, or int8).
    Returns a dict with float64 ``k_cache`` / ``ckv_cache`` (int64 codes for
    int8 caches; untouched slots decoded from the input), the pre-rounding
    values ``k_pre`` / ``ckv_pre`` (NaN where nothing was written), the boolean
    ``k_written`` / ``ckv_written`` slot masks, ``k_rope`` / ``c_kv`` (float64,
    when is_output_kv) and ``bad_index`` (count of out-of-range slots).
    """
    x_all = decode_bf16(kv)
    B, N, S, Dkv = x_all.shape
    R = rope_size
    if variant == 1:
        rms_size = Dkv - R
    elif variant == 2:
        rms_size = Dkv
    else:
        raise ValueError("variant must be 1 or 2")

    # (1) RmsNorm
    x = x_all[..., :rms_size]
    y = rms_norm(x, decode_bf16(gamma), epsilon)

    # (2) interleaved RoPE
    xr = x_all[..., rms_size:] if variant == 1 else y[..., :R]
    y_rope = interleave_rope(xr, decode_bf16(cos), decode_bf16(sin))
    rope_out = y_rope if variant == 1 else np.concatenate([y_rope, y[..., R:]], axis=-1)
    v_src = y if variant == 1 else decode_bf16(v)

    # (3) Quant
    per_head = variant == 2
    k_val, k_pre = quantize(rope_out, k_scale, k_offset, per_head)
    c_val, c_pre = quantize(v_src, v_scale, v_offset, per_head)

    # (4) Scatter
    def start(cache, quant):
        if quant:
            return np.asarray(cache).astype(np.int64), np.full(cache.shape, np.nan)
        return decode_bf16(cache), None

    k_out, k_pre_out = start(k_cache, k_scale is not None)
    c_out, c_pre_out = start(ckv_cache, v_scale is not None)
    k_written = np.zeros(k_out.shape, dtype=bool)
    c_written = np.zeros(c_out.shape, dtype=bool)
    slots = k_out.shape[0] * block_size
    idx = np.asarray(index, dtype=np.int64)
    tok = np.nonzero((idx >= 0) & (idx < slots))[0]
    bad = int(np.count_nonzero((idx != -1) & ((idx < -1) | (idx >= slots))))
    b, s = tok // S, tok % S
    blk, off = idx[tok] // block_size, idx[tok] % block_size

    def put(dst, src, mask, pre_dst, pre_src):
        if cache_mode == "PA_BNSD":      # [block_num, N, block_size, D]
            dst[blk, :, off, :] = src[b, :, s, :]
            mask[blk, :, off, :] = True
            if pre_dst is not None:
                pre_dst[blk, :, off, :] = pre_src[b, :, s, :]
        elif cache_mode == "PA":         # [block_num, block_size, N, D]
            dst[blk, off, :, :] = src[b, :, s, :]
            mask[blk, off, :, :] = True
            if pre_dst is not None:
                pre_dst[blk, off, :, :] = pre_src[b, :, s, :]
        else:
            raise ValueError(cache_mode)

    put(k_out, k_val, k_written, k_pre_out, k_pre)
    put(c_out, c_val, c_written, c_pre_out, c_pre)

    res = {"k_cache": k_out, "ckv_cache": c_out, "k_pre": k_pre_out, "ckv_pre": c_pre_out,
           "k_written": k_written, "ckv_written": c_written, "bad_index": bad}
    # (5) optional outputs
    if is_output_kv:
        res["k_rope"] = rope_out
        res["c_kv"] = v_src
    return res
