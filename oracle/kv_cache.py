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

Cache modes (cache/index constraint table):
  * Norm: caches [B, N, Scache, D]; index [B, S] holds each token's offset in its
    batch's cache, -1 = skip; values may repeat across batches.
  * PA / PA_BNSD: token index as above.
  * PA_BLK_BNSD: caches as PA_BNSD; index [B * ceil(S / block_size)] holds the
    start slot of each block of block_size tokens (-1 = skip the block); token s
    of batch b goes to slot index[b, s // block_size] + s % block_size.
  Out-of-range slots are neither written nor trapped; they are counted.
Outputs (5) exist in every PA mode; in Norm mode only for V2 with quantisation
(the "Norm" row of the input-combination table); V1 in Norm mode takes no
quantisation parameters.
cos/sin may be [B, N, 1, R], broadcast over S (the "S-axis broadcast" of the
input-combination table).  Inputs are bf16 or fp16 (the parameter table); a
non-quantised cache has the input's dtype.  A quantised cache is int8 (formula
(3)) or FP8 E4M3 / E5M2: for FP8 the reading is the same x * scale + offset,
rounded to the nearest FP8 value (ties to even) and saturated at the largest
finite value, in place of round().clamp(-128, 127).

Quant scales/offsets are per channel: shape [D] for V1, [N, D] for V2.
Values are computed in float64; bf16 caches receive the unrounded value (the
comparison applies the bf16 tolerance), int8 caches receive the int code, and
the pre-rounding value of every code is returned for the tie rule.
"""
from __future__ import annotations

import numpy as np

from .codes import decode_bf16, decode_fp16, encode_fp8


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


def quantize(x: np.ndarray, scale, offset, n_axis_param: bool, qtype: str = "int8"):
    """Returns (value, pre_round).  ``value`` is int64 codes when a scale is given
    (int8 values, or the FP8 code bytes for qtype "e4m3" / "e5m2")."""
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
    if qtype == "int8":
        return np.clip(np.rint(v), -128, 127).astype(np.int64), v
    return encode_fp8(v, qtype).astype(np.int64), v


def token_slots(index, cache_mode: str, b: np.ndarray, s: np.ndarray, S: int, block_size: int) -> np.ndarray:
    """Slot of each token (b, s) from ``index``, per the cache/index constraint
    table: the token's own entry (Norm: an offset in batch b's cache; PA modes: a
    slot of the paged cache), or for PA_BLK_BNSD its block's start slot plus its
    position in the block.  -1 = skip; -2 marks an illegal negative block start."""
    idx = np.asarray(index, dtype=np.int64).reshape(-1)
    if cache_mode in ("Norm", "PA", "PA_BNSD"):
        return idx[b * S + s]
    if cache_mode == "PA_BLK_BNSD":
        nb = -(-S // block_size)
        first = idx[b * nb + s // block_size]
        return np.where(first == -1, -1, np.where(first < -1, -2, first + s % block_size))
    raise ValueError(cache_mode)


def cache_rows(cache_mode: str, b: np.ndarray, p: np.ndarray, block_size: int):
    """Index of the (all-heads) cache rows of token slots p: Norm [B, N, Scache, D]
    at (b, :, p); PA_BNSD / PA_BLK_BNSD [block_num, N, block_size, D] at
    (p // block_size, :, p % block_size); PA [block_num, block_size, N, D] at
    (p // block_size, p % block_size)."""
    if cache_mode == "Norm":
        return (b, slice(None), p)
    if cache_mode in ("PA_BNSD", "PA_BLK_BNSD"):
        return (p // block_size, slice(None), p % block_size)
    return (p // block_size, p % block_size)


def kv_rms_norm_rope_cache(kv, gamma, cos, sin, index, k_cache, ckv_cache, *, variant: int,
                           rope_size: int, block_size: int, cache_mode: str = "PA_BNSD",
                           epsilon: float = 1e-5, k_scale=None, k_offset=None, v_scale=None,
                           v_offset=None, v=None, is_output_kv: bool = False, dtype: str = "bf16",
                           k_qtype: str = "int8", v_qtype: str = "int8") -> dict:
    """Run the operator on host arrays.

    kv, gamma, cos, sin, v: bf16 or fp16 bit patterns (uint16), ``dtype``.  index:
    int64 (shape per cache mode, see the module docstring).  k_cache / ckv_cache: the
    caches before the call (uint16 bit patterns, int8 values, or uint8 FP8 codes).
    Returns a dict with float64 ``k_cache`` / ``ckv_cache`` (int64 codes for
    quantised caches; untouched slots decoded from the input), the pre-rounding
    values ``k_pre`` / ``ckv_pre`` (NaN where nothing was written), the boolean
    ``k_written`` / ``ckv_written`` slot masks, ``k_rope`` / ``c_kv`` (float64,
    when they are output) and ``bad_index`` (count of out-of-range slots).
    """
    dec = {"bf16": decode_bf16, "fp16": decode_fp16}[dtype]
    x_all = dec(kv)
    B, N, S, Dkv = x_all.shape
    R = rope_size
    if variant == 1:
        rms_size = Dkv - R
    elif variant == 2:
        rms_size = Dkv
    else:
        raise ValueError("variant must be 1 or 2")
    quant = k_scale is not None or v_scale is not None
    if cache_mode == "Norm" and variant == 1 and quant:
        raise ValueError("V1 in Norm mode takes no quantisation parameters")

    # (1) RmsNorm
    x = x_all[..., :rms_size]
    y = rms_norm(x, dec(gamma), epsilon)

    # (2) interleaved RoPE (cos/sin [B, N, S or 1, R] broadcast over S)
    xr = x_all[..., rms_size:] if variant == 1 else y[..., :R]
    y_rope = interleave_rope(xr, dec(cos), dec(sin))
    rope_out = y_rope if variant == 1 else np.concatenate([y_rope, y[..., R:]], axis=-1)
    v_src = y if variant == 1 else dec(v)

    # (3) Quant
    per_head = variant == 2
    k_val, k_pre = quantize(rope_out, k_scale, k_offset, per_head, k_qtype)
    c_val, c_pre = quantize(v_src, v_scale, v_offset, per_head, v_qtype)

    # (4) Scatter: for every token (b, s) the cache row of head n, or none
    def start(cache, q):
        if q:
            return np.asarray(cache).astype(np.int64), np.full(cache.shape, np.nan)
        return dec(cache), None

    k_out, k_pre_out = start(k_cache, k_scale is not None)
    c_out, c_pre_out = start(ckv_cache, v_scale is not None)
    k_written = np.zeros(k_out.shape, dtype=bool)
    c_written = np.zeros(c_out.shape, dtype=bool)
    limit = k_out.shape[2] if cache_mode == "Norm" else k_out.shape[0] * block_size
    bb, ss = np.meshgrid(np.arange(B), np.arange(S), indexing="ij")
    bb, ss = bb.reshape(-1), ss.reshape(-1)  # token t = b * S + s
    p = token_slots(index, cache_mode, bb, ss, S, block_size)
    ok = (p >= 0) & (p < limit)
    bad = int(np.count_nonzero((p != -1) & ~ok))
    tok = np.nonzero(ok)[0]
    b, s_, pt = bb[tok], ss[tok], p[tok]
    at = cache_rows(cache_mode, b, pt, block_size)

    def put(dst, src, mask, pre_dst, pre_src):
        dst[at] = src[b, :, s_]
        mask[at] = True
        if pre_dst is not None:
            pre_dst[at] = pre_src[b, :, s_]

    put(k_out, k_val, k_written, k_pre_out, k_pre)
    put(c_out, c_val, c_written, c_pre_out, c_pre)

    res = {"k_cache": k_out, "ckv_cache": c_out, "k_pre": k_pre_out, "ckv_pre": c_pre_out,
           "k_written": k_written, "ckv_written": c_written, "bad_index": bad}
    # (5) optional outputs
    if is_output_kv and (cache_mode != "Norm" or (variant == 2 and quant)):
        res["k_rope"] = rope_out
        res["c_kv"] = v_src
    return res
