"""Seeded synthetic inputs for the attention prologue.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds input generation only: shapes, random draws, the FP8/MX/bf16 encoding
of those draws, and the RoPE cos/sin tables.  None of the arithmetic that the
two operators perform (projection, norm, rotation, quantisation, scatter)
lives here.

Every tensor is drawn from ``numpy.random.default_rng([seed, k])`` with one
sub-stream ``k`` per tensor, so any tensor can be regenerated on its own.

Workloads (stand-ins for the pages' Wan2.2-A14B DiT attention and the
DeepSeek-V3 MLA KV cache; no dataset or checkpoint is used):

* ``qkv_tiny``      fused QKV self-attention, S=128, H=256, n_q=n_kv=2, d=64.
* ``qkv_wan480``    Wan2.2-A14B 480p self-attention, S=32760 (21x30x52), H=5120,
                    40 heads, d=128, I=15360, 3-D RoPE.
* ``qkv_wan_cross`` Wan2.2-A14B cross-attention: Q from S=32760 image tokens,
                    K and V from L=512 text tokens, separate 5120-wide calls.
* ``kv_mla_v1``     KvRmsNormRopeCache V1, kv [32,1,4096,576], PA_BNSD bs=128.
* ``qkv_wan720``    Wan2.2-A14B 720p self-attention, S=75600 (21x45x80), plus
* ``kv_sep_v2``     KvRmsNormRopeCache V2, kv [8,8,4096,192], v [8,8,4096,128].
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

E4M3_MAX = 448.0


def stream(seed: int, k: int) -> np.random.Generator:
    """Independent PCG64 sub-stream ``k`` of workload ``seed``."""
    return np.random.default_rng([seed, k])


# ---------------------------------------------------------------------------
# Wan2.2 latent grid (vLLM-Omni-Neuron "Context Parallelism", section
# "Sequence Length Constraints": latent frames (F-1)//4+1, patch grid
# (H//8)//2 x (W//8)//2).
# ---------------------------------------------------------------------------
def wan_latent_grid(num_frames: int, height: int, width: int) -> tuple[int, int, int]:
    return ((num_frames - 1) // 4 + 1, (height // 8) // 2, (width // 8) // 2)


# ---------------------------------------------------------------------------
# Encoders (input preparation).  FP8 E4M3 uses torch's float8_e4m3fn cast
# (round-to-nearest-even); bf16 uses torch's bfloat16 cast (RNE).
# ---------------------------------------------------------------------------
def encode_e4m3(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def encode_fp16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def encode_bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def row_quantize_e4m3(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Row-scaled FP8 activation: one fp32 scale per row = max(amax, 1e-30)/448."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=1)
    scale = (np.maximum(amax, np.float32(1e-30)) / np.float32(E4M3_MAX)).astype(np.float32)
    codes = encode_e4m3(x / scale[:, None])
    return codes, scale


def mx_quantize_e4m3(w: np.ndarray, block: int = 32) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8 weight [H, I]: e4m3 codes plus a ue8m0 exponent per (32-row H block, column).

    Exponent e = clamp(ceil(log2(amax/448)) + 127, 0, 254); an all-zero block gets 127.
    """
    w = np.asarray(w, dtype=np.float32)
    H, I = w.shape
    assert H % block == 0
    blocks = w.reshape(H // block, block, I)
    amax = np.max(np.abs(blocks), axis=1).astype(np.float64)  # [H/32, I]
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.ceil(np.log2(amax / E4M3_MAX)) + 127, 127)
    e = np.clip(e, 0, 254)
    # guard against log2 rounding: the scaled block must fit in e4m3
    over = (amax / np.exp2(e - 127)) > E4M3_MAX
    e = np.where(over & (e < 254), e + 1, e).astype(np.uint8)
    scale = np.exp2(e.astype(np.float64) - 127).astype(np.float32)
    codes = encode_e4m3((blocks / scale[:, None, :]).reshape(H, I))
    return codes, e


# ---------------------------------------------------------------------------
# RoPE tables
# ---------------------------------------------------------------------------
def rope_rotate_half_1d(positions: np.ndarray, d: int, theta: float = 10000.0):
    """Rotate-half cos/sin [len(positions), d]: lanes j and j+d/2 share angle pos*theta^(-2j/d)."""
    j = np.arange(d // 2, dtype=np.float64)
    freq = theta ** (-2.0 * j / d)
    ang = positions.astype(np.float64)[:, None] * freq[None, :]
    ang = np.concatenate([ang, ang], axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope_rotate_half_3d(grid: tuple[int, int, int], d: int, theta: float = 10000.0):
    """Wan-style 3-D rotate-half cos/sin [f*h*w, d].

    The d/2 frequency pairs are split over (frame, height, width) as
    d/2 - 2*(d//6), d//6, d//6 pairs (22/21/21 for d=128); each axis uses its own
    ladder theta^(-2j/d_axis) with d_axis = 2*pairs.  Token t sits at
    f = t // (h*w), y = (t // w) % h, x = t % w.
    """
    F, Hh, Ww = grid
    n_hw = d // 6
    pairs = [d // 2 - 2 * n_hw, n_hw, n_hw]
    t = np.arange(F * Hh * Ww, dtype=np.int64)
    pos = [t // (Hh * Ww), (t // Ww) % Hh, t % Ww]
    angs = []
    for p, npairs in zip(pos, pairs):
        d_axis = 2 * npairs
        j = np.arange(npairs, dtype=np.float64)
        freq = theta ** (-2.0 * j / d_axis)
        angs.append(p.astype(np.float64)[:, None] * freq[None, :])
    ang = np.concatenate(angs, axis=1)  # [T, d/2]
    ang = np.concatenate([ang, ang], axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope_interleaved_table(S: int, R: int, theta: float = 10000.0):
    """cos/sin rows [S, R] for the interleaved op: cos[j] = cos[j+R/2] = cos(s*theta^(-2j/R))."""
    j = np.arange(R // 2, dtype=np.float64)
    freq = theta ** (-2.0 * j / R)
    ang = np.arange(S, dtype=np.float64)[:, None] * freq[None, :]
    ang = np.concatenate([ang, ang], axis=1)
    return np.cos(ang), np.sin(ang)


# ---------------------------------------------------------------------------
# Fused QKV projection inputs
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class QKVCase:
    name: str
    B: int
    S: int
    H: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    a: np.ndarray            # [T, H] uint8 e4m3
    a_scale: np.ndarray      # [T] fp32
    w: np.ndarray            # [H, I] uint8 e4m3
    w_block_exp: np.ndarray  # [H/32, I] uint8 ue8m0
    weight_scales: np.ndarray | None  # [I] fp32 or None
    bias: np.ndarray | None  # [I] uint16 (bf16 bits) or None
    q_norm: bool | str      # False, True (across heads) or "per_head"
    k_norm: bool | str
    fused_rope: bool
    cos: np.ndarray | None   # [T, d] fp32
    sin: np.ndarray | None
    q_gamma: np.ndarray | None  # [num_heads*d] fp32 ([d] for the per-head norm)
    k_gamma: np.ndarray | None  # [num_kv_heads*d] fp32 ([d] for the per-head norm)
    eps: float

    @property
    def T(self) -> int:
        return self.B * self.S

    @property
    def I(self) -> int:
        return (self.num_heads + 2 * self.num_kv_heads) * self.head_dim

    @property
    def flops(self) -> float:
        return 2.0 * self.T * self.H * self.I


def make_qkv(name: str, seed: int, S: int, H: int, num_heads: int, num_kv_heads: int,
             head_dim: int, *, B: int = 1, rope: str | None = "1d", grid=None,
             q_norm: bool | str = True, k_norm: bool | str = True, bias: bool = True,
             weight_scales: bool = False, eps: float = 1e-6,
             a_std: float = 1.0, w_std: float = 0.02) -> QKVCase:
    T = B * S
    I = (num_heads + 2 * num_kv_heads) * head_dim
    a32 = stream(seed, 0).standard_normal((T, H), dtype=np.float32) * np.float32(a_std)
    a, a_scale = row_quantize_e4m3(a32)
    del a32
    w32 = stream(seed, 1).standard_normal((H, I), dtype=np.float32) * np.float32(w_std)
    w, w_exp = mx_quantize_e4m3(w32)
    del w32
    b = encode_bf16(stream(seed, 2).normal(0.0, 0.01, I).astype(np.float32)) if bias else None
    ws = stream(seed, 3).uniform(0.5, 2.0, I).astype(np.float32) if weight_scales else None
    qn = head_dim if q_norm == "per_head" else num_heads * head_dim
    kn = head_dim if k_norm == "per_head" else num_kv_heads * head_dim
    qg = stream(seed, 4).uniform(0.5, 1.5, qn).astype(np.float32) if q_norm else None
    kg = (stream(seed, 5).uniform(0.5, 1.5, kn).astype(np.float32)
          if (k_norm and num_kv_heads > 0) else None)
    cos = sin = None
    if rope == "1d":
        pos = np.tile(np.arange(S), B)
        cos, sin = rope_rotate_half_1d(pos, head_dim)
    elif rope == "3d":
        assert grid is not None and grid[0] * grid[1] * grid[2] == S
        c1, s1 = rope_rotate_half_3d(grid, head_dim)
        cos, sin = np.tile(c1, (B, 1)), np.tile(s1, (B, 1))
    return QKVCase(name, B, S, H, num_heads, num_kv_heads, head_dim, a, a_scale, w, w_exp,
                   ws, b, q_norm, k_norm if num_kv_heads > 0 else False, rope is not None, cos, sin,
                   qg, kg, eps)


def qkv_tiny(seed: int = 0) -> QKVCase:
    """S=128, H=256, n_q=n_kv=2, d=64, I=384, 1-D RoPE positions 0..127."""
    return make_qkv("qkv_tiny", seed, S=128, H=256, num_heads=2, num_kv_heads=2, head_dim=64)


def qkv_wan_self(seed: int, grid: tuple[int, int, int], name: str) -> QKVCase:
    S = grid[0] * grid[1] * grid[2]
    return make_qkv(name, seed, S=S, H=5120, num_heads=40, num_kv_heads=40, head_dim=128,
                    rope="3d", grid=grid)


def qkv_wan480(seed: int = 1) -> QKVCase:
    """Wan2.2-A14B 480p self-attention: 81 frames at 480x832 -> grid 21x30x52, S=32760."""
    return qkv_wan_self(seed, wan_latent_grid(81, 480, 832), "qkv_wan480")


def qkv_wan720(seed: int = 4) -> QKVCase:
    """Wan2.2-A14B 720p self-attention: 81 frames at 720x1280 -> grid 21x45x80, S=75600."""
    return qkv_wan_self(seed, wan_latent_grid(81, 720, 1280), "qkv_wan720")


def hidden_bf16(seed: int, T: int, H: int, *, k: int = 20, rows_per_chunk: int = 4096) -> np.ndarray:
    """bf16 hidden state [T, H] (bit patterns) for the row quantiser: N(0,1) entries,
    a per-row factor 2^U(-3,3), and 1 % of the channels (a fixed set) scaled by 8,
    the outlier channels of transformer activations.  Generated in row chunks so
    that full-size inputs need little host memory."""
    g = stream(seed, k)
    outliers = g.choice(H, max(1, H // 100), replace=False)
    col = np.ones(H, np.float32)
    col[outliers] = 8.0
    out = np.empty((T, H), np.uint16)
    for r0 in range(0, T, rows_per_chunk):
        r1 = min(T, r0 + rows_per_chunk)
        x = g.standard_normal((r1 - r0, H), dtype=np.float32)
        x *= np.exp2(g.uniform(-3, 3, (r1 - r0, 1))).astype(np.float32) * col[None, :]
        out[r0:r1] = encode_bf16(x)
    return out


def qkv_wan_cross(seed: int = 2) -> list[QKVCase]:
    """Wan2.2-A14B cross-attention: three single-segment calls (num_kv_heads=0).

    Q: S=32760 image tokens, normed, no RoPE.  K: L=512 text tokens, normed.
    V: L=512 text tokens, no norm.
    """
    S = 32760
    q = make_qkv("cross_q", seed * 10 + 0, S=S, H=5120, num_heads=40, num_kv_heads=0,
                 head_dim=128, rope=None)
    k = make_qkv("cross_k", seed * 10 + 1, S=512, H=5120, num_heads=40, num_kv_heads=0,
                 head_dim=128, rope=None)
    v = make_qkv("cross_v", seed * 10 + 2, S=512, H=5120, num_heads=40, num_kv_heads=0,
                 head_dim=128, rope=None, q_norm=False)
    return [q, k, v]


def sample_rows(T: int, seed: int, n_head: int = 128, n_tail: int = 256, n_rand: int = 640) -> np.ndarray:
    """Deterministic row sample: first n_head rows, last n_tail rows, n_rand random rows."""
    rows = set(range(min(n_head, T)))
    rows.update(range(max(0, T - n_tail), T))
    if T > 0:
        rows.update(stream(seed, 99).choice(T, size=min(n_rand, T), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


# ---------------------------------------------------------------------------
# KvRmsNormRopeCache inputs
# ---------------------------------------------------------------------------
CACHE_MODES = {"Norm": 0, "PA": 1, "PA_BNSD": 2, "PA_BLK_BNSD": 4}


@dataclasses.dataclass
class KVCase:
    name: str
    variant: int
    B: int
    N: int
    S: int
    Dkv: int
    Dv: int
    rope_size: int
    kv: np.ndarray           # [B,N,S,Dkv] uint16 bf16 bits
    gamma: np.ndarray        # [rms_size] uint16
    cos: np.ndarray          # [B,N,S,R] uint16
    sin: np.ndarray
    index: np.ndarray        # [B*S] int64
    cache_mode: str
    block_num: int
    block_size: int
    k_cache: np.ndarray      # initial cache contents (sentinel), uint16 or int8
    ckv_cache: np.ndarray
    k_scale: np.ndarray | None
    k_offset: np.ndarray | None
    v_scale: np.ndarray | None
    v_offset: np.ndarray | None
    v: np.ndarray | None     # [B,N,S,Dv] uint16 (V2)
    eps: float
    is_output_kv: bool
    dtype: str = "bf16"       # kv / gamma / cos / sin / v (and non-quantised caches): bf16 or fp16
    k_qtype: str = "int8"     # quantised k cache: int8, e4m3 or e5m2
    v_qtype: str = "int8"
    cache_seq: int = 0        # Norm mode: Scache

    @property
    def rope_broadcast(self) -> bool:
        return self.cos.shape[2] == 1 and self.S > 1

    @property
    def rms_size(self) -> int:
        return self.Dkv - self.rope_size if self.variant == 1 else self.Dkv

    @property
    def k_width(self) -> int:
        return self.rope_size if self.variant == 1 else self.Dkv

    @property
    def ckv_width(self) -> int:
        return self.rms_size if self.variant == 1 else self.Dv

    def algorithmic_bytes(self) -> int:
        rows = self.B * self.N * self.S
        b = self.kv.nbytes + self.cos.nbytes + self.sin.nbytes + self.index.nbytes + self.gamma.nbytes
        if self.v is not None:
            b += self.v.nbytes
        if self.cache_mode == "PA_BLK_BNSD":
            starts = self.index.reshape(self.B, -1)
            s_blk = np.arange(self.S) // self.block_size
            valid = int(np.count_nonzero(starts[:, s_blk] >= 0)) * self.N
        else:
            valid = int(np.count_nonzero(self.index >= 0)) * self.N
        kb = 1 if self.k_scale is not None else 2
        cb = 1 if self.v_scale is not None else 2
        b += valid * (self.k_width * kb + self.ckv_width * cb)
        quant = self.k_scale is not None or self.v_scale is not None
        if self.is_output_kv and (self.cache_mode != "Norm" or (self.variant == 2 and quant)):
            b += rows * (self.k_width + self.ckv_width) * 2
        for p in (self.k_scale, self.k_offset, self.v_scale, self.v_offset):
            if p is not None:
                b += p.nbytes
        return b


K_SENTINEL_BF16 = 0x7FBF  # a bf16 NaN pattern the op never writes
K_SENTINEL_FP16 = 0x7FBF  # an fp16 NaN pattern the op never writes
K_SENTINEL_I8 = -77
K_SENTINEL_FP8 = 0x7F     # NaN in both E4M3 and E5M2


def make_kv(name: str, seed: int, *, variant: int, B: int, N: int, S: int, Dkv: int, Dv: int,
            rope_size: int = 64, block_size: int = 128, block_num: int | None = None,
            cache_mode: str = "PA_BNSD", quant_k: bool = False, quant_v: bool = False,
            offsets: bool = True, with_v: bool | None = None, eps: float = 1e-5,
            is_output_kv: bool = True, skip_frac: float = 0.0, dtype: str = "bf16",
            k_qtype: str = "int8", v_qtype: str = "int8", rope_broadcast: bool = False,
            cache_seq: int | None = None, k_scalar: bool = False, v_scalar: bool = False) -> KVCase:
    """Synthetic KvRmsNormRopeCache call.

    kv, v ~ N(0,1); gamma ~ U(0.5,1.5); cos/sin from position s with ladder
    theta=1e4 (same values for every b and n; with ``rope_broadcast`` one row
    [B, N, 1, R] at position S-1, broadcast over S); all of them in ``dtype``
    (bf16 or fp16).  index, per ``cache_mode``:
      PA / PA_BNSD: the first B*S entries of a random permutation of the
        block_num*block_size slots;
      Norm: per batch, the first S entries of a random permutation of the
        cache_seq (Scache) offsets, shape [B, S];
      PA_BLK_BNSD: per block of block_size tokens, the start slot of a distinct
        random cache block (block id * block_size), shape [B * ceil(S / block_size)];
    a fraction ``skip_frac`` of the entries replaced by -1.  Quant scales
    ~ U(10,40), offsets ~ U(-2,2), per channel ([D] in V1, [N, D] in V2) or, with
    ``k_scalar`` / ``v_scalar`` (V1), one value [1] for the whole component; a
    quantised cache is int8 or FP8 (``k_qtype``, ``v_qtype``).  Caches start
    filled with a sentinel the op never writes.
    """
    enc = {"bf16": encode_bf16, "fp16": encode_fp16}[dtype]
    rms = Dkv - rope_size if variant == 1 else Dkv
    kw = rope_size if variant == 1 else Dkv
    cw = rms if variant == 1 else Dv
    nb = -(-S // block_size)
    if block_num is None:
        block_num = B * nb if cache_mode == "PA_BLK_BNSD" else -(-B * S // block_size)
    if cache_mode == "Norm" and cache_seq is None:
        cache_seq = S
    kv = enc(stream(seed, 0).standard_normal((B, N, S, Dkv), dtype=np.float32))
    gamma = enc(stream(seed, 1).uniform(0.5, 1.5, rms).astype(np.float32))
    c, s = rope_interleaved_table(S, rope_size)
    rows = slice(S - 1, S) if rope_broadcast else slice(0, S)
    srope = 1 if rope_broadcast else S
    cos = np.broadcast_to(enc(c[rows].astype(np.float32)), (B, N, srope, rope_size)).copy()
    sin = np.broadcast_to(enc(s[rows].astype(np.float32)), (B, N, srope, rope_size)).copy()
    g2 = stream(seed, 2)
    if cache_mode in ("PA", "PA_BNSD"):
        index = g2.permutation(block_num * block_size)[: B * S].astype(np.int64)
    elif cache_mode == "Norm":
        index = np.stack([g2.permutation(cache_seq)[:S] for _ in range(B)]).astype(np.int64)
    elif cache_mode == "PA_BLK_BNSD":
        index = (g2.permutation(block_num)[: B * nb] * block_size).astype(np.int64)
    else:
        raise ValueError(cache_mode)
    if skip_frac > 0:
        drop = stream(seed, 3).random(index.shape) < skip_frac
        index[drop] = -1
    v = None
    if with_v if with_v is not None else (variant == 2):
        v = enc(stream(seed, 4).standard_normal((B, N, S, Dv), dtype=np.float32))
    qshape_k = ((1,) if k_scalar else (kw,)) if variant == 1 else (N, kw)
    qshape_v = ((1,) if v_scalar else (cw,)) if variant == 1 else (N, cw)
    ks = stream(seed, 5).uniform(10, 40, qshape_k).astype(np.float32) if quant_k else None
    ko = stream(seed, 6).uniform(-2, 2, qshape_k).astype(np.float32) if (quant_k and offsets) else None
    vs = stream(seed, 7).uniform(10, 40, qshape_v).astype(np.float32) if quant_v else None
    vo = stream(seed, 8).uniform(-2, 2, qshape_v).astype(np.float32) if (quant_v and offsets) else None
    if cache_mode in ("PA_BNSD", "PA_BLK_BNSD"):
        kshape, cshape = (block_num, N, block_size, kw), (block_num, N, block_size, cw)
    elif cache_mode == "PA":
        kshape, cshape = (block_num, block_size, N, kw), (block_num, block_size, N, cw)
    else:  # Norm
        kshape, cshape = (B, N, cache_seq, kw), (B, N, cache_seq, cw)

    def cache(shape, quant, qtype):
        if not quant:
            return np.full(shape, K_SENTINEL_BF16 if dtype == "bf16" else K_SENTINEL_FP16, np.uint16)
        if qtype == "int8":
            return np.full(shape, K_SENTINEL_I8, np.int8)
        return np.full(shape, K_SENTINEL_FP8, np.uint8)

    return KVCase(name, variant, B, N, S, Dkv, Dv, rope_size, kv, gamma, cos, sin, index,
                  cache_mode, block_num, block_size, cache(kshape, quant_k, k_qtype),
                  cache(cshape, quant_v, v_qtype), ks, ko, vs, vo, v, eps, is_output_kv,
                  dtype, k_qtype, v_qtype, cache_seq or 0)


def kv_mla_v1(seed: int = 3, quant: bool = False) -> KVCase:
    """DeepSeek-V3 MLA combined kv: [32,1,4096,576], norm on 512, RoPE on 64, PA_BNSD bs=128."""
    return make_kv("kv_mla_v1" + ("_int8" if quant else "_bf16"), seed, variant=1, B=32, N=1,
                   S=4096, Dkv=576, Dv=512, block_size=128, block_num=1024,
                   quant_k=quant, quant_v=quant, is_output_kv=True)


def kv_sep_v2(seed: int = 4, is_output_kv: bool = False) -> KVCase:
    """Separate k/v: kv [8,8,4096,192], v [8,8,4096,128], int8 per-head quant, PA_BNSD bs=128."""
    return make_kv("kv_sep_v2", seed, variant=2, B=8, N=8, S=4096, Dkv=192, Dv=128,
                   block_size=128, block_num=256, quant_k=True, quant_v=True,
                   is_output_kv=is_output_kv)
