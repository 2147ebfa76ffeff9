"""Pins for the fp64 oracle (CPU only).

Each check ties an oracle function to something other than itself: a library
routine (torch's float8/bfloat16 casts, torch.nn.functional.rms_norm, numpy
complex multiplication, torch integer matmul, torch.round), a closed form
(one-hot / permutation projections, power-of-two scales), an invariant of the
method (RoPE inverse and norm preservation), values fixed by hand in
``tests/golden/hand_values.txt``, or brute force over a tiny scatter.

The ``check_*`` helpers raise AssertionError on a mismatch; ``test_mutants``
plants plausible mistakes in the oracle (sign flips, transposed operands,
wrong widths, dropped terms) and confirms that some check catches each one.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import codes, kv_cache as okv, qkv_cte as oq, row_quant as orq
from rope_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def torch_e4m3(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).view(torch.float8_e4m3fn).to(F64).numpy()


def torch_bf16(b):
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).to(F64).numpy()


def torch_fp16(b):
    return torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.float16).to(F64).numpy()


def finite_e4m3_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    return np.where((c & 0x7F) == 0x7F, np.uint8(0x38), c)


def assert_close(got, exp, rtol=1e-12, atol=1e-12):
    np.testing.assert_allclose(np.asarray(got, np.float64), np.asarray(exp, np.float64), rtol=rtol, atol=atol)


# ---------------------------------------------------------------------------
# code decoders
# ---------------------------------------------------------------------------
def check_decoders():
    allc = np.arange(256, dtype=np.uint8)
    got, exp = codes.decode_e4m3(allc), torch_e4m3(allc)
    assert np.array_equal(np.isnan(got), np.isnan(exp))
    assert np.array_equal(got[~np.isnan(got)], exp[~np.isnan(exp)])
    got = codes.decode_ue8m0(allc)
    exp = torch.from_numpy(allc).view(torch.float8_e8m0fnu).to(F64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(exp))
    assert np.array_equal(got[~np.isnan(got)], exp[~np.isnan(exp)])
    bits = np.random.default_rng(7).integers(0, 65536, 4096).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite patterns
    assert np.array_equal(codes.decode_bf16(bits), torch_bf16(bits))


def test_decoders_match_torch_casts():
    check_decoders()


def test_e4m3_spec_points():
    # OCP FP8 E4M3: 0x38 = 1.0, 0x7E = 448 (max), 0x08 = 2^-6 (min normal), 0x01 = 2^-9, 0xB8 = -1
    v = codes.decode_e4m3(np.array([0x38, 0x7E, 0x08, 0x01, 0xB8, 0x00, 0x80], np.uint8))
    assert list(v) == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, -1.0, 0.0, 0.0]
    assert np.isnan(codes.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()


# ---------------------------------------------------------------------------
# projection
# ---------------------------------------------------------------------------
def check_projection_permutation():
    """W is a non-symmetric permutation: O[t, pi(h)] = A_hat[t, h]."""
    rng = np.random.default_rng(1)
    T, H = 6, 64
    a = finite_e4m3_codes(rng, (T, H))
    a_scale = np.exp2(rng.integers(-3, 4, T)).astype(np.float32)
    pi = (np.arange(H) * 5 + 3) % H
    w = np.zeros((H, H), np.uint8)
    w[np.arange(H), pi] = 0x38
    w_exp = np.full((H // 32, H), 127, np.uint8)
    got = oq.project(a, a_scale, w, w_exp)
    exp = np.zeros((T, H))
    exp[:, pi] = torch_e4m3(a) * a_scale[:, None]
    assert_close(got, exp, 0, 0)


def check_projection_block_scales():
    """One-hot rows pick W_hat's row h; the block scale of row h is e[h // 32, i]."""
    rng = np.random.default_rng(2)
    H, I = 96, 40
    hs = np.array([0, 31, 32, 63, 64, 95, 17, 70])
    a = np.zeros((len(hs), H), np.uint8)
    a[np.arange(len(hs)), hs] = 0x38
    w = np.full((H, I), 0x38, np.uint8)
    w_exp = rng.integers(120, 135, (H // 32, I)).astype(np.uint8)
    ws = rng.uniform(0.5, 2.0, I).astype(np.float32)
    got = oq.project(a, np.ones(len(hs), np.float32), w, w_exp, weight_scales=ws)
    exp = np.exp2(w_exp[hs // 32, :].astype(np.float64) - 127) * ws.astype(np.float64)[None, :]
    assert_close(got, exp, 0, 0)


def check_projection_integer_exact():
    """Small integer codes, unit scales: the product is an exact integer matmul."""
    rng = np.random.default_rng(3)
    T, H, I = 9, 64, 48
    table = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48}
    ai = rng.integers(-4, 5, (T, H))
    wi = rng.integers(-4, 5, (H, I))
    enc = lambda m: np.vectorize(lambda v: table[abs(v)] | (0x80 if v < 0 else 0))(m).astype(np.uint8)
    bias_bits = synth.encode_bf16(rng.integers(-8, 9, I).astype(np.float32))
    got = oq.project(enc(ai), np.ones(T, np.float32), enc(wi), np.full((H // 32, I), 127, np.uint8),
                     bias=bias_bits)
    exp = (torch.from_numpy(ai) @ torch.from_numpy(wi)).numpy() + torch_bf16(bias_bits)[None, :]
    assert_close(got, exp, 0, 0)


def check_projection_scaling():
    """Row scales and channel scales factor out; zero activations give the bias."""
    rng = np.random.default_rng(4)
    T, H, I = 5, 64, 32
    a = finite_e4m3_codes(rng, (T, H))
    w = finite_e4m3_codes(rng, (H, I))
    e = rng.integers(118, 136, (H // 32, I)).astype(np.uint8)
    base = oq.project(a, np.ones(T, np.float32), w, e)
    k = rng.integers(-4, 5, T)
    c = np.exp2(rng.integers(-3, 4, I)).astype(np.float32)
    got = oq.project(a, np.exp2(k).astype(np.float32), w, e, weight_scales=c)
    assert_close(got, base * np.exp2(k)[:, None] * c[None, :], 0, 0)
    bias = synth.encode_bf16(rng.normal(0, 1, I).astype(np.float32))
    z = oq.project(np.zeros((T, H), np.uint8), np.ones(T, np.float32), w, e, bias=bias)
    assert_close(z, np.broadcast_to(torch_bf16(bias), (T, I)), 0, 0)


@pytest.mark.parametrize("check", [check_projection_permutation, check_projection_block_scales,
                                   check_projection_integer_exact, check_projection_scaling])
def test_projection(check):
    check()


# ---------------------------------------------------------------------------
# across-heads RMSNorm + rotate-half RoPE
# ---------------------------------------------------------------------------
def read_hand_values():
    rows = []
    with open(os.path.join(GOLDEN, "hand_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            lhs, rhs = line.split("|")
            kind, *args = lhs.split()
            rows.append((kind, [float(x) for x in args], [float(x) for x in rhs.split()]))
    return rows


def check_rmsnorm_hand():
    for kind, args, out in read_hand_values():
        if kind == "rmsnorm":
            x = np.array([args])
            assert_close(oq.rms_norm_across_heads(x, np.ones(2), 0.0), [out], 1e-15, 0)
            assert_close(okv.rms_norm(x, np.ones(2), 0.0), [out], 1e-15, 0)


def test_rmsnorm_hand_value():
    check_rmsnorm_hand()


def complex_rope_rotate_half(y, theta, d):
    """Rotate-half pairs (j, j+d/2) as complex numbers y_j + i*y_{j+d/2} times the unit
    number ``theta`` (an angle array, or complex cos + i*sin values)."""
    T = y.shape[0]
    yh = y.reshape(T, -1, d)
    rot = theta if np.iscomplexobj(theta) else np.exp(1j * theta)
    z = (yh[..., : d // 2] + 1j * yh[..., d // 2:]) * rot[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1).reshape(T, -1)


def complex_rope_interleaved(x, theta):
    """Interleaved pairs (2j, 2j+1) as complex numbers, output de-interleaved (reals first)."""
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def identity_qkv(nq, nkv, d, T, seed, rope):
    """A case whose projection is known without the oracle: H = I, W = identity, unit scales."""
    rng = np.random.default_rng(seed)
    I = (nq + 2 * nkv) * d
    a = finite_e4m3_codes(rng, (T, I))
    a_scale = np.exp2(rng.integers(-2, 3, T)).astype(np.float32)
    w = np.zeros((I, I), np.uint8)
    w[np.arange(I), np.arange(I)] = 0x38
    e = np.full((I // 32, I), 127, np.uint8)
    bias = synth.encode_bf16(rng.normal(0, 0.5, I).astype(np.float32))
    qg = rng.uniform(0.5, 1.5, nq * d).astype(np.float32)
    kg = rng.uniform(0.5, 1.5, nkv * d).astype(np.float32) if nkv else None
    theta = rng.uniform(-np.pi, np.pi, (T, d // 2))
    cos = np.concatenate([np.cos(theta)] * 2, axis=1).astype(np.float32)
    sin = np.concatenate([np.sin(theta)] * 2, axis=1).astype(np.float32)
    # the fp32 tables are not exactly unit-modulus: rotate by the complex number cos + i*sin
    theta = cos[:, : d // 2].astype(np.float64) + 1j * sin[:, : d // 2].astype(np.float64)
    o = torch_e4m3(a) * a_scale[:, None] + torch_bf16(bias)[None, :]
    kw = dict(num_heads=nq, num_kv_heads=nkv, head_dim=d, bias=bias, q_gamma=qg, k_gamma=kg,
              eps=1e-6, fused_rope=rope, cos=cos if rope else None, sin=sin if rope else None)
    return a, a_scale, w, e, kw, o, theta, (cos, sin)


def torch_rms(x, g, eps):
    return F.rms_norm(torch.from_numpy(x), (x.shape[1],), torch.from_numpy(np.asarray(g, np.float64)), eps).numpy()


def check_qkv_norm_segments():
    """No RoPE: Q and K are F.rms_norm over their own widths (n_q != n_kv), V is O."""
    nq, nkv, d = 3, 2, 32
    a, s, w, e, kw, o, _, _ = identity_qkv(nq, nkv, d, 7, 5, rope=False)
    got = oq.qkv_cte_mx(a, s, w, e, **kw)
    qw, kwid = nq * d, nkv * d
    assert_close(got[:, :qw], torch_rms(o[:, :qw], kw["q_gamma"], 1e-6), 1e-12, 1e-13)
    assert_close(got[:, qw:qw + kwid], torch_rms(o[:, qw:qw + kwid], kw["k_gamma"], 1e-6), 1e-12, 1e-13)
    assert_close(got[:, qw + kwid:], o[:, qw + kwid:], 0, 0)


def check_qkv_single_segment():
    """num_kv_heads = 0: the whole width is normed as Q."""
    a, s, w, e, kw, o, _, _ = identity_qkv(4, 0, 32, 5, 6, rope=False)
    got = oq.qkv_cte_mx(a, s, w, e, **kw)
    assert_close(got, torch_rms(o, kw["q_gamma"], 1e-6), 1e-12, 1e-13)


def check_qkv_norm_then_rope():
    """With RoPE: complex rotation of F.rms_norm(segment) (gamma before rotation); V untouched."""
    nq, nkv, d = 2, 3, 64
    a, s, w, e, kw, o, theta, _ = identity_qkv(nq, nkv, d, 6, 7, rope=True)
    got = oq.qkv_cte_mx(a, s, w, e, **kw)
    qw, kwid = nq * d, nkv * d
    exp_q = complex_rope_rotate_half(torch_rms(o[:, :qw], kw["q_gamma"], 1e-6), theta, d)
    exp_k = complex_rope_rotate_half(torch_rms(o[:, qw:qw + kwid], kw["k_gamma"], 1e-6), theta, d)
    assert_close(got[:, :qw], exp_q, 1e-9, 1e-12)
    assert_close(got[:, qw:qw + kwid], exp_k, 1e-9, 1e-12)
    assert_close(got[:, qw + kwid:], o[:, qw + kwid:], 0, 0)


def check_rotate_half_invariants():
    rng = np.random.default_rng(8)
    T, n, d = 5, 3, 16
    y = rng.normal(0, 1, (T, n * d))
    theta = rng.uniform(-3, 3, (T, d // 2))
    cos = np.concatenate([np.cos(theta)] * 2, axis=1)
    sin = np.concatenate([np.sin(theta)] * 2, axis=1)
    r = oq.rope_rotate_half(y, cos, sin, d)
    assert_close(r, complex_rope_rotate_half(y, theta, d), 1e-12, 1e-14)
    assert_close(oq.rope_rotate_half(r, cos, -sin, d), y, 1e-12, 1e-14)          # inverse
    assert_close(oq.rope_rotate_half(y, np.ones_like(cos), np.zeros_like(sin), d), y, 0, 0)
    yh, rh = y.reshape(T, n, d), r.reshape(T, n, d)                              # pair norms
    assert_close(np.hypot(rh[..., : d // 2], rh[..., d // 2:]), np.hypot(yh[..., : d // 2], yh[..., d // 2:]), 1e-12, 1e-14)


@pytest.mark.parametrize("check", [check_qkv_norm_segments, check_qkv_single_segment,
                                   check_qkv_norm_then_rope, check_rotate_half_invariants])
def test_qkv(check):
    check()


# ---------------------------------------------------------------------------
# KvRmsNormRopeCache
# ---------------------------------------------------------------------------
def check_interleave_rope():
    rng = np.random.default_rng(9)
    R = 16
    x = rng.normal(0, 1, (4, 3, R))
    theta = rng.uniform(-3, 3, (4, 3, R // 2))
    cos = np.concatenate([np.cos(theta)] * 2, axis=-1)
    sin = np.concatenate([np.sin(theta)] * 2, axis=-1)
    r = okv.interleave_rope(x, cos, sin)
    assert_close(r, complex_rope_interleaved(x, theta), 1e-12, 1e-14)
    # the interleaved form equals rotate-half applied to the de-interleaved vector
    deint = np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)
    assert_close(r.reshape(12, R), oq.rope_rotate_half(deint.reshape(12, R), cos.reshape(12, R), sin.reshape(12, R), R), 1e-12, 1e-14)
    # inverse: rotate-half with -sin on the output, then re-interleave
    back = oq.rope_rotate_half(r.reshape(12, R), cos.reshape(12, R), -sin.reshape(12, R), R).reshape(4, 3, R)
    re = np.empty_like(x)
    re[..., 0::2], re[..., 1::2] = back[..., : R // 2], back[..., R // 2:]
    assert_close(re, x, 1e-12, 1e-14)
    # position 0 (cos 1, sin 0) is the de-interleave permutation
    assert_close(okv.interleave_rope(x, np.ones_like(cos), np.zeros_like(sin)), deint, 0, 0)


def check_quant_hand():
    for kind, args, out in read_hand_values():
        if kind == "quant":
            x, sc, of = args
            q, pre = okv.quantize(np.array([x]), np.array([sc]), np.array([of]), False)
            assert int(q[0]) == int(out[0]), (x, sc, of, q)
            t = torch.round(torch.tensor([x * sc + of], dtype=F64)).clamp(-128, 127)
            assert int(t[0]) == int(out[0])


def tiny_kv(variant, cache_mode="PA_BNSD", quant=False, seed=11):
    if variant == 1:
        kw = dict(B=2, N=1, S=5, Dkv=24, Dv=16, rope_size=8)
    else:
        kw = dict(B=2, N=2, S=5, Dkv=24, Dv=16, rope_size=8)
    case = synth.make_kv("tiny", seed, variant=variant, block_size=4, block_num=4,
                         cache_mode=cache_mode, quant_k=quant, quant_v=quant, skip_frac=0.3, **kw)
    case.index[1] = -1
    return case


def run_kv(case):
    return okv.kv_rms_norm_rope_cache(
        case.kv, case.gamma, case.cos, case.sin, case.index, case.k_cache, case.ckv_cache,
        variant=case.variant, rope_size=case.rope_size, block_size=case.block_size,
        cache_mode=case.cache_mode, epsilon=case.eps, k_scale=case.k_scale, k_offset=case.k_offset,
        v_scale=case.v_scale, v_offset=case.v_offset, v=case.v, is_output_kv=True,
        dtype=case.dtype, k_qtype=case.k_qtype, v_qtype=case.v_qtype)


def expected_kv_rows(case):
    """Per (b, n, s) rows built from library routines: F.rms_norm, complex rotation, torch.round."""
    dec = torch_bf16 if case.dtype == "bf16" else torch_fp16
    x = dec(case.kv)
    B, N, S, Dkv = x.shape
    R = case.rope_size
    rms = case.rms_size
    g = torch.from_numpy(dec(case.gamma))
    y = F.rms_norm(torch.from_numpy(x[..., :rms].copy()), (rms,), g, case.eps).numpy()
    cos, sin = dec(case.cos), dec(case.sin)
    theta = np.arctan2(sin[..., : R // 2], cos[..., : R // 2])
    radius = np.hypot(sin[..., : R // 2], cos[..., : R // 2])  # bf16 tables are not exactly unit
    def rot(v):
        z = (v[..., 0::2] + 1j * v[..., 1::2]) * radius * np.exp(1j * theta)
        return np.concatenate([z.real, z.imag], axis=-1)
    if case.variant == 1:
        k_rows, c_rows = rot(x[..., rms:]), y
    else:
        k_rows, c_rows = np.concatenate([rot(y[..., :R]), y[..., R:]], axis=-1), dec(case.v)

    def q(v, sc, of):
        if sc is None:
            return v, None
        sc = sc if case.variant == 1 else sc[None, :, None, :]
        pre = torch.from_numpy(v) * torch.from_numpy(np.asarray(sc, np.float64))
        if of is not None:
            of = of if case.variant == 1 else of[None, :, None, :]
            pre = pre + torch.from_numpy(np.asarray(of, np.float64))
        return torch.round(pre).clamp(-128, 127).numpy(), pre.numpy()

    kq, kpre = q(k_rows, case.k_scale, case.k_offset)
    cq, cpre = q(c_rows, case.v_scale, case.v_offset)
    return k_rows, c_rows, kq, kpre, cq, cpre


def check_kv_op(variant, cache_mode, quant):
    case = tiny_kv(variant, cache_mode, quant)
    res = run_kv(case)
    k_rows, c_rows, kq, kpre, cq, cpre = expected_kv_rows(case)
    B, N, S = case.B, case.N, case.S
    assert_close(res["k_rope"], k_rows, 1e-12, 1e-12)
    assert_close(res["c_kv"], c_rows, 1e-12, 1e-12)
    k_exp = torch_bf16(case.k_cache) if not quant else case.k_cache.astype(np.float64)
    c_exp = torch_bf16(case.ckv_cache) if not quant else case.ckv_cache.astype(np.float64)
    k_exp, c_exp = k_exp.copy(), c_exp.copy()
    kp_exp = np.full(k_exp.shape, np.nan)
    cp_exp = np.full(c_exp.shape, np.nan)
    seen = set()
    for b in range(B):                       # brute-force scatter
        for s in range(S):
            p = int(case.index[b * S + s])
            if p == -1:
                continue
            assert p not in seen
            seen.add(p)
            blk, off = divmod(p, case.block_size)
            for n in range(N):
                kr = kq[b, n, s] if quant else k_rows[b, n, s]
                cr = cq[b, n, s] if quant else c_rows[b, n, s]
                at = (blk, n, off) if cache_mode == "PA_BNSD" else (blk, off, n)
                k_exp[at], c_exp[at] = kr, cr
                if quant:
                    kp_exp[at], cp_exp[at] = kpre[b, n, s], cpre[b, n, s]
    assert_close(res["k_cache"], k_exp, 1e-12, 1e-12)
    assert_close(res["ckv_cache"], c_exp, 1e-12, 1e-12)
    assert res["k_written"].sum() == len(seen) * N * case.k_width
    if quant:
        assert_close(res["k_pre"], kp_exp, 1e-12, 1e-12)
        assert_close(res["ckv_pre"], cp_exp, 1e-12, 1e-12)


def check_kv_v1_bf16():
    check_kv_op(1, "PA_BNSD", False)


def check_kv_v1_int8():
    check_kv_op(1, "PA_BNSD", True)


def check_kv_v2_int8():
    check_kv_op(2, "PA_BNSD", True)


def check_kv_v2_pa_bf16():
    check_kv_op(2, "PA", False)


def check_kv_bad_index():
    case = tiny_kv(2, "PA_BNSD", False)
    case.index[0] = case.block_num * case.block_size  # out of range: counted, not written
    case.index[2] = -5
    res = run_kv(case)
    assert res["bad_index"] == 2
    valid = np.count_nonzero(case.index >= 0) - 1
    assert res["k_written"].sum() == valid * case.N * case.k_width


@pytest.mark.parametrize("check", [check_interleave_rope, check_quant_hand, check_kv_v1_bf16,
                                   check_kv_v1_int8, check_kv_v2_int8, check_kv_v2_pa_bf16,
                                   check_kv_bad_index])
def test_kv(check):
    check()


# ---------------------------------------------------------------------------
# generator fixtures fixed by the pages
# ---------------------------------------------------------------------------
def test_wan_seq_len_golden():
    with open(os.path.join(GOLDEN, "wan_seq_len.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            fr, h, w, lf, ph, pw, st = map(int, line.split())
            assert synth.wan_latent_grid(fr, h, w) == (lf, ph, pw)
            assert lf * ph * pw == st


def test_generator_encodings():
    """Row scale bounds every code to |x| <= 448; MX exponents keep blocks in range."""
    c = synth.qkv_tiny()
    a_hat = torch_e4m3(c.a)
    assert np.nanmax(np.abs(a_hat)) <= 448 and not np.isnan(a_hat).any()
    assert np.allclose(np.max(np.abs(a_hat), axis=1), 448, rtol=0.07)
    w_hat = torch_e4m3(c.w)
    assert not np.isnan(w_hat).any() and np.max(np.abs(w_hat)) <= 448


# ---------------------------------------------------------------------------
# row FP8 quantisation (qkv_cte page, Interface: row-packed activation)
# ---------------------------------------------------------------------------
def _torch_e4m3_code(v):
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def check_e4m3_encoder_vs_torch():
    """The encoder agrees with torch's float8_e4m3fn cast (round-half-even) on every
    representable value, every midpoint between neighbours, and random values."""
    mags = codes.decode_e4m3(np.arange(127, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2  # exact in fp32: at most 5 significant bits
    rng = np.random.default_rng(11)
    vals = np.concatenate([mags, mids, rng.uniform(-448, 448, 20000), rng.normal(0, 0.01, 5000),
                           np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 2.0 ** -9 * 1.5])])
    vals = np.concatenate([vals, -vals]).astype(np.float32)
    assert np.array_equal(orq.encode_e4m3_rne_sat(vals), _torch_e4m3_code(vals))


def check_e4m3_encoder_saturates():
    """Magnitudes above the largest finite value (448) saturate to it, keeping the sign."""
    big = np.array([448.0001, 464.0, 479.9, 480.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(orq.encode_e4m3_rne_sat(big) == 0x7E)
    assert np.all(orq.encode_e4m3_rne_sat(-big) == 0xFE)


def check_row_quant_hand():
    """x = [1, -2, 0.5, 0, ...]: amax 2, inv 224, products [224, -448, 112, 0]:
    codes 0.1110.110, 1.1111.110, 0.1101.110, 0; scale = 2 / 448 in fp32."""
    x = np.zeros((1, 16), np.float32)
    x[0, :4] = [1.0, -2.0, 0.5, 0.0]
    c, sc = orq.row_quantize(synth.encode_bf16(x))
    assert list(c[0, :4]) == [0x76, 0xFE, 0x6E, 0x00] and not c[0, 4:].any()
    assert sc.dtype == np.float32 and sc[0] == np.float32(2.0) / np.float32(448.0)


def check_row_quant_zero_row():
    """A row of zeros: zero codes with the input's sign, scale 2^-100 / 448; a row of
    bf16 subnormals (amax below the 2^-100 floor) stays finite and small."""
    x = np.zeros((2, 16), np.float32)
    bits = synth.encode_bf16(x)
    bits[1, 5] = 0x8000  # -0.0
    c, sc = orq.row_quantize(bits)
    assert np.all(sc == np.float32(2.0 ** -100) / np.float32(448))
    expect = np.zeros((2, 16), np.uint8)
    expect[1, 5] = 0x80
    assert np.array_equal(c, expect)
    sub = np.zeros((1, 16), np.uint16)
    sub[0, :3] = [0x0001, 0x8040, 0x007F]  # subnormal bf16 values, |x| < 2^-126
    c, sc = orq.row_quantize(sub)
    assert np.isfinite(sc).all() and not np.any((c & 0x7F) == 0x7F)
    assert np.all((c & 0x7F) <= 0x08)  # tiny codes: |x| * 448 * 2^100 < 2^-6


def check_row_quant_roundtrip():
    """Dequantised codes reproduce x: the row maximum maps to +-448 exactly, and every
    value in E4M3's normal range is within half a unit of its 3-bit mantissa."""
    rng = np.random.default_rng(12)
    x = (rng.normal(0, 1, (32, 512)) * np.exp2(rng.integers(-12, 12, 32))[:, None]).astype(np.float32)
    bits = synth.encode_bf16(x)
    xb = codes.decode_bf16(bits)
    c, sc = orq.row_quantize(bits)
    y = codes.decode_e4m3(c) * sc.astype(np.float64)[:, None]
    amax = np.max(np.abs(xb), axis=1)
    i = np.argmax(np.abs(xb), axis=1)
    assert np.all((c[np.arange(32), i] & 0x7F) == 0x7E)
    normal = np.abs(xb) * (448.0 / amax)[:, None] >= 2.0 ** -6
    rel = np.abs(y - xb)[normal] / np.abs(xb)[normal]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-5)
    assert np.allclose(sc, amax / 448.0, rtol=2 ** -23, atol=0)


def _rn_binary32(v):
    """Exact round-to-nearest-even of a Fraction to IEEE binary32 (normal and subnormal
    range, no overflow at these sizes), returned as a Fraction."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** max(e - 23, -149)     # 24 significant bits, or the subnormal step
    q, r = divmod(a, quantum)
    if r * 2 > quantum or (r * 2 == quantum and q % 2 == 1):
        q += 1
    return sign * q * quantum


def _e4m3_code_exact(v):
    """E4M3 code of a Fraction by exhaustive search over the format's definition (bias 7,
    3 mantissa bits, no infinities, S.1111.111 = NaN): nearest magnitude, ties to the even
    code, above 448 saturated to 448, the sign bit from v."""
    from fractions import Fraction
    mags = []
    for code in range(127):                        # 0x00 .. 0x7E, increasing magnitude
        ef, mf = code >> 3, code & 7
        mags.append(Fraction(mf, 8) * Fraction(2) ** -6 if ef == 0 else (1 + Fraction(mf, 8)) * Fraction(2) ** (ef - 7))
    a = min(abs(v), mags[-1])
    best = min(range(127), key=lambda c: (abs(mags[c] - a), c % 2))
    return best | (0x80 if v < 0 else 0)


def check_row_quant_exact_rational():
    """The row quantiser against exact rational arithmetic: scale = RN32(m / 448) and
    code = E4M3(RN32(x / scale)) evaluated with Fractions and an independent binary32
    rounding, on rows of bf16 values whose largest magnitudes span 2^-20 .. 2^20.  On
    this input the multiply-by-reciprocal form E4M3(RN32(x * RN32(448 / m))) gives other
    codes (checked with plain float32 arithmetic), so the pin tells the readings apart."""
    from fractions import Fraction
    rng = np.random.default_rng(19)  # a seed whose rows hold codes the two forms round apart
    x = (rng.normal(0, 1, (48, 96)) * np.exp2(rng.integers(-20, 20, 48))[:, None]).astype(np.float32)
    bits = synth.encode_bf16(x)
    xb = codes.decode_bf16(bits).astype(np.float32)
    c, sc = orq.row_quantize(bits)
    for t in range(xb.shape[0]):
        m = max(max(Fraction(float(v)) for v in np.abs(xb[t])), Fraction(2) ** -100)
        scale = _rn_binary32(m / 448)
        assert Fraction(float(sc[t])) == scale, t
        for h in range(xb.shape[1]):
            q = _rn_binary32(Fraction(float(xb[t, h])) / scale)
            assert c[t, h] == _e4m3_code_exact(q), (t, h, float(xb[t, h]), float(q))
    m32 = np.maximum(np.max(np.abs(xb), axis=1), np.float32(2.0 ** -100)).astype(np.float32)
    recip = orq.encode_e4m3_rne_sat((xb * (np.float32(448) / m32)[:, None]).astype(np.float32))
    assert np.count_nonzero(recip != c) > 0


def check_row_quant_packed():
    """The packed row: H codes, then the fp32 scale's four bytes."""
    rng = np.random.default_rng(13)
    bits = synth.encode_bf16(rng.normal(0, 3, (5, 48)).astype(np.float32))
    pk = orq.row_quantize_packed(bits)
    c, sc = orq.row_quantize(bits)
    assert pk.shape == (5, 52) and np.array_equal(pk[:, :48], c)
    assert np.array_equal(np.ascontiguousarray(pk[:, 48:]).view("<f4").ravel(), sc)


@pytest.mark.parametrize("check", [check_e4m3_encoder_vs_torch, check_e4m3_encoder_saturates,
                                   check_row_quant_hand, check_row_quant_zero_row,
                                   check_row_quant_roundtrip, check_row_quant_packed,
                                   check_row_quant_exact_rational])
def test_row_quant(check):
    check()


def check_nbsd_layout():
    """NBSd puts token (b, s)'s head h at [h, b, s, :]: checked against an
    explicit index formula on a tensor whose entries encode their position."""
    B, S, d, n = 2, 3, 4, 5
    out = np.arange(B * S * n * d, dtype=np.float64).reshape(B * S, n * d)
    r = oq.to_nbsd(out, B, S, d)
    assert r.shape == (n, B, S, d)
    for h in range(n):
        for b in range(B):
            for s_ in range(S):
                for j in range(d):
                    assert r[h, b, s_, j] == (b * S + s_) * n * d + h * d + j


def test_nbsd_layout():
    check_nbsd_layout()


# ---------------------------------------------------------------------------
# KvRmsNormRopeCache variants: Norm and PA_BLK_BNSD cache modes, S-broadcast
# cos/sin, fp16 inputs, FP8 caches
# ---------------------------------------------------------------------------
TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def torch_fp8_code(v, fmt):
    return torch.from_numpy(np.ascontiguousarray(v, np.float64)).to(TORCH_FP8[fmt]).view(torch.uint8) \
        .numpy().astype(np.int64)


def check_fp8_encoders_vs_torch():
    """encode_fp8 agrees with torch's float8 casts (round-half-even) on every finite
    value, every midpoint between neighbours and random values, and saturates."""
    rng = np.random.default_rng(21)
    for fmt, top in (("e4m3", 0x7F), ("e5m2", 0x7C)):
        dec = codes.decode_e4m3 if fmt == "e4m3" else codes.decode_e5m2
        mags = dec(np.arange(top, dtype=np.uint8))
        mids = (mags[:-1] + mags[1:]) / 2
        vals = np.concatenate([mags, mids, rng.uniform(-FP8_MAX[fmt], FP8_MAX[fmt], 20000),
                               rng.normal(0, 0.05, 5000)])
        vals = np.concatenate([vals, -vals])
        assert np.array_equal(codes.encode_fp8(vals, fmt).astype(np.int64), torch_fp8_code(vals, fmt)), fmt
        big = np.array([FP8_MAX[fmt] * 1.01, FP8_MAX[fmt] * 1.2, 1e9])
        assert np.all(codes.encode_fp8(big, fmt) == top - 1) and np.all(codes.encode_fp8(-big, fmt) == 0x80 | (top - 1))


def brute_scatter(case, k_rows, c_rows):
    """Per-token loops over the cache/index constraint table: the expected caches
    (float64 values or codes) and the number of written (token, head) rows."""
    dec = codes.decode_bf16 if case.dtype == "bf16" else codes.decode_fp16
    k_exp = dec(case.k_cache) if case.k_scale is None else case.k_cache.astype(np.float64)
    c_exp = dec(case.ckv_cache) if case.v_scale is None else case.ckv_cache.astype(np.float64)
    k_exp, c_exp = k_exp.copy(), c_exp.copy()
    B, N, S, bs = case.B, case.N, case.S, case.block_size
    nb = -(-S // bs)
    written = 0
    for b in range(B):
        for s_ in range(S):
            if case.cache_mode == "Norm":
                p = int(case.index[b, s_])
                if not 0 <= p < case.cache_seq:
                    continue
                at = [(b, n, p) for n in range(N)]
            else:
                if case.cache_mode == "PA_BLK_BNSD":
                    first = int(case.index[b * nb + s_ // bs])
                    if first < 0:
                        continue
                    p = first + s_ % bs
                else:
                    p = int(case.index[b * S + s_])
                if not 0 <= p < case.block_num * bs:
                    continue
                blk, off = divmod(p, bs)
                at = [(blk, off, n) if case.cache_mode == "PA" else (blk, n, off) for n in range(N)]
            for n, a in enumerate(at):
                k_exp[a], c_exp[a] = k_rows[b, n, s_], c_rows[b, n, s_]
                written += 1
    return k_exp, c_exp, written


def quant_rows(case, rows, scale, offset, qtype):
    if scale is None:
        return rows
    sc = scale if case.variant == 1 else scale[None, :, None, :]
    pre = torch.from_numpy(rows) * torch.from_numpy(np.asarray(sc, np.float64))
    if offset is not None:
        of = offset if case.variant == 1 else offset[None, :, None, :]
        pre = pre + torch.from_numpy(np.asarray(of, np.float64))
    if qtype == "int8":
        return torch.round(pre).clamp(-128, 127).numpy()
    m = FP8_MAX[qtype]
    return torch_fp8_code(pre.clamp(-m, m).numpy(), qtype).astype(np.float64)


def check_kv_mode(case, expect_outputs=True):
    res = run_kv(case)
    k_rows, c_rows, *_ = expected_kv_rows(case)
    kq = quant_rows(case, k_rows, case.k_scale, case.k_offset, case.k_qtype)
    cq = quant_rows(case, c_rows, case.v_scale, case.v_offset, case.v_qtype)
    k_exp, c_exp, written = brute_scatter(case, kq, cq)
    assert_close(res["k_cache"], k_exp, 1e-12, 1e-12)
    assert_close(res["ckv_cache"], c_exp, 1e-12, 1e-12)
    assert res["k_written"].sum() == written * case.k_width
    assert ("k_rope" in res) == expect_outputs
    return res


def check_kv_norm_mode():
    """Norm mode: caches [B, N, Scache, D], index [B, S] of per-batch offsets (values
    repeat across batches); V2 with int8 quantisation writes k_rope / c_kv."""
    case = synth.make_kv("norm", 31, variant=2, B=2, N=2, S=5, Dkv=24, Dv=16, rope_size=8,
                         cache_mode="Norm", cache_seq=7, quant_k=True, quant_v=True, skip_frac=0.2)
    case.index[1, :] = case.index[0, :]  # the same offsets in another batch are legal
    case.index[0, 2] = 7                 # out of range: counted, not written
    res = check_kv_mode(case)
    assert res["bad_index"] == 1


def check_kv_norm_v1_no_outputs():
    """Norm mode, V1, no quantisation: the caches are written, k_rope / c_kv are not."""
    case = synth.make_kv("norm1", 32, variant=1, B=2, N=1, S=5, Dkv=24, Dv=16, rope_size=8,
                         cache_mode="Norm", cache_seq=6, skip_frac=0.2)
    check_kv_mode(case, expect_outputs=False)


def check_kv_blk_mode():
    """PA_BLK_BNSD: one start slot per block of block_size tokens; a skipped block
    skips all its tokens; the last block of a batch may be partial."""
    case = synth.make_kv("blk", 33, variant=2, B=2, N=2, S=10, Dkv=24, Dv=16, rope_size=8,
                         block_size=4, block_num=8, cache_mode="PA_BLK_BNSD")
    case.index[1] = -1
    check_kv_mode(case)


def check_kv_rope_broadcast():
    """cos/sin [B, N, 1, R] act as that row repeated along S."""
    case = synth.make_kv("bc", 34, variant=2, B=2, N=2, S=5, Dkv=24, Dv=16, rope_size=8,
                         block_size=4, block_num=4, rope_broadcast=True, quant_k=True)
    assert case.cos.shape[2] == 1
    res = run_kv(case)
    rep = dataclasses.replace(case, cos=np.repeat(case.cos, case.S, axis=2), sin=np.repeat(case.sin, case.S, axis=2))
    res2 = run_kv(rep)
    for key in ("k_cache", "ckv_cache", "k_rope", "c_kv"):
        assert np.array_equal(res[key], res2[key], equal_nan=True), key
    check_kv_mode(case)


def check_kv_fp16_inputs():
    """fp16 inputs whose values bf16 also holds exactly give the same result as bf16."""
    rng = np.random.default_rng(35)
    base = synth.make_kv("f16", 35, variant=2, B=2, N=2, S=5, Dkv=24, Dv=16, rope_size=8,
                         block_size=4, block_num=4)
    def grid(shape, lo, hi):  # multiples of 1/16: exact in both formats
        return (rng.integers(int(lo * 16), int(hi * 16) + 1, shape) / 16).astype(np.float32)
    half = base.cos.shape[:-1] + (base.rope_size // 2,)
    dup = lambda h: np.concatenate([h, h], axis=-1)  # cos[j] = cos[j + R/2], as the tables are built
    vals = dict(kv=grid(base.kv.shape, -4, 4), gamma=grid(base.gamma.shape, 0.5, 1.5),
                cos=dup(grid(half, -1, 1)), sin=dup(grid(half, -1, 1)), v=grid(base.v.shape, -4, 4))
    b16 = dataclasses.replace(base, **{k: synth.encode_bf16(x) for k, x in vals.items()})
    f16 = dataclasses.replace(base, dtype="fp16", k_cache=np.full(base.k_cache.shape, 0x7FBF, np.uint16),
                              ckv_cache=np.full(base.ckv_cache.shape, 0x7FBF, np.uint16),
                              **{k: synth.encode_fp16(x) for k, x in vals.items()})
    r16, rb = run_kv(f16), run_kv(b16)
    for key in ("k_rope", "c_kv"):
        assert np.array_equal(r16[key], rb[key]), key
    check_kv_mode(f16)


def check_kv_fp8_caches():
    """k cache E4M3, ckv cache E5M2: the codes are torch's float8 casts of the
    saturated x * scale + offset."""
    case = synth.make_kv("fp8", 36, variant=2, B=2, N=2, S=5, Dkv=24, Dv=16, rope_size=8,
                         block_size=4, block_num=4, quant_k=True, quant_v=True, k_qtype="e4m3",
                         v_qtype="e5m2", skip_frac=0.2)
    case.k_scale *= 20.0  # reach the E4M3 saturation point on some channels
    check_kv_mode(case)


def check_kv_scalar_quant_params():
    """V1 quantisation parameters of shape [1] (the page's shape table): the same
    caches as [D] arrays filled with that value, and every written int8 code is
    torch's round(x * s + o).clamp(-128, 127) of the unquantised output."""
    case = synth.make_kv("scal", 39, variant=1, B=2, N=1, S=6, Dkv=24, Dv=16, rope_size=8,
                         block_size=4, block_num=4, quant_k=True, quant_v=True, skip_frac=0.2,
                         k_scalar=True, v_scalar=True)
    assert case.k_scale.shape == (1,) and case.v_offset.shape == (1,)
    got = run_kv(case)
    full = dataclasses.replace(case, k_scale=np.full(8, case.k_scale[0], np.float32),
                               k_offset=np.full(8, case.k_offset[0], np.float32),
                               v_scale=np.full(16, case.v_scale[0], np.float32),
                               v_offset=np.full(16, case.v_offset[0], np.float32))
    ref = run_kv(full)
    for key in ("k_cache", "ckv_cache"):
        assert np.array_equal(got[key], ref[key]), key
    for cache, out, sc, of, written in (("k_cache", "k_rope", case.k_scale, case.k_offset, "k_written"),
                                        ("ckv_cache", "c_kv", case.v_scale, case.v_offset, "ckv_written")):
        x = torch.from_numpy(got[out])                                       # [B, N, S, D]
        codes = torch.round(x * float(sc[0]) + float(of[0])).clamp(-128, 127).to(torch.int64)
        p = okv.token_slots(case.index, "PA_BNSD", np.repeat(np.arange(2), 6), np.tile(np.arange(6), 2), 6, 4)
        for t, slot in enumerate(p):
            if slot < 0:
                continue
            b, s_ = divmod(t, 6)
            row = got[cache][slot // 4, 0, slot % 4]
            assert np.array_equal(row, codes[b, 0, s_].numpy()), (cache, t)
        assert got[written].sum() > 0


@pytest.mark.parametrize("check", [check_fp8_encoders_vs_torch, check_kv_norm_mode, check_kv_norm_v1_no_outputs,
                                   check_kv_blk_mode, check_kv_rope_broadcast, check_kv_fp16_inputs,
                                   check_kv_fp8_caches, check_kv_scalar_quant_params])
def test_kv_variants(check):
    check()


def check_per_head_norm():
    """Per-head qk-norm = torch's rms_norm over each head's d_head slice with the
    [d_head] gamma; with one head it equals the across-heads norm."""
    rng = np.random.default_rng(37)
    T, n, d = 5, 3, 16
    x = rng.normal(0, 2, (T, n * d))
    g = rng.uniform(0.5, 1.5, d)
    got = oq.rms_norm_per_head(x, g, 1e-6, d)
    exp = F.rms_norm(torch.from_numpy(x.reshape(T, n, d)), (d,), torch.from_numpy(g), 1e-6).numpy().reshape(T, -1)
    assert_close(got, exp, 1e-12, 1e-12)
    one = oq.rms_norm_per_head(x[:, :d], g, 1e-6, d)
    assert_close(one, oq.rms_norm_across_heads(x[:, :d], g, 1e-6), 1e-12, 1e-12)


def check_qkv_per_head_segments():
    """qkv_cte_mx with per-head norms: Q and K each per head, then RoPE; V untouched."""
    c = synth.make_qkv("ph", 38, S=20, H=256, num_heads=2, num_kv_heads=2, head_dim=64)
    qg, kg = c.q_gamma[:64], c.k_gamma[:64]
    got = oq.qkv_cte_mx(c.a, c.a_scale, c.w, c.w_block_exp, num_heads=2, num_kv_heads=2, head_dim=64,
                        bias=c.bias, q_norm="per_head", k_norm="per_head", q_gamma=qg, k_gamma=kg,
                        eps=c.eps, fused_rope=True, cos=c.cos, sin=c.sin)
    o = oq.project(c.a, c.a_scale, c.w, c.w_block_exp, bias=c.bias)
    ref = o.copy()
    for lo, g in ((0, qg), (128, kg)):
        seg = o[:, lo:lo + 128].reshape(20, 2, 64)
        y = F.rms_norm(torch.from_numpy(seg), (64,), torch.from_numpy(g.astype(np.float64)), c.eps).numpy()
        ref[:, lo:lo + 128] = oq.rope_rotate_half(y.reshape(20, 128), c.cos, c.sin, 64)
    assert_close(got, ref, 1e-12, 1e-12)


@pytest.mark.parametrize("check", [check_per_head_norm, check_qkv_per_head_segments])
def test_per_head(check):
    check()


# ---------------------------------------------------------------------------
# planted mistakes: every mutant must be caught by at least one check
# ---------------------------------------------------------------------------
ALL_CHECKS = [check_decoders, check_projection_permutation, check_projection_block_scales,
              check_projection_integer_exact, check_projection_scaling, check_rmsnorm_hand,
              check_qkv_norm_segments, check_qkv_single_segment, check_qkv_norm_then_rope,
              check_rotate_half_invariants, check_interleave_rope, check_quant_hand,
              check_kv_v1_bf16, check_kv_v1_int8, check_kv_v2_int8, check_kv_v2_pa_bf16,
              check_kv_bad_index, check_e4m3_encoder_vs_torch, check_e4m3_encoder_saturates,
              check_row_quant_hand, check_row_quant_zero_row, check_row_quant_roundtrip,
              check_row_quant_packed, check_row_quant_exact_rational, check_nbsd_layout, check_fp8_encoders_vs_torch,
              check_kv_norm_mode, check_kv_norm_v1_no_outputs, check_kv_blk_mode,
              check_kv_rope_broadcast, check_kv_fp16_inputs, check_kv_fp8_caches,
              check_per_head_norm, check_qkv_per_head_segments]


def mutants():
    orig_rh = oq.rope_rotate_half
    orig_norm = oq.rms_norm_across_heads
    orig_dw = oq.dequant_weight
    orig_il = okv.interleave_rope
    orig_q = okv.quantize
    orig_e4 = codes.decode_e4m3
    orig_kvn = okv.rms_norm

    def rh_sign(y, cos, sin, d):            # sin sign flipped
        return orig_rh(y, cos, -sin, d)

    def norm_no_eps(x, g, eps):             # eps dropped
        return orig_norm(x, g, 0.0)

    def norm_pre_gamma_width(x, g, eps):    # divide by the wrong width
        return orig_norm(x, g, eps) * np.sqrt(x.shape[1] / (x.shape[1] + 32))

    def dw_transposed_blocks(w, e, ws=None):  # block index taken along I instead of H
        H, I = w.shape
        ee = np.repeat(e, 32, axis=0)[:H]
        ee = np.roll(ee, 1, axis=1)
        return orig_e4(w) * np.exp2(ee.astype(np.float64) - 127) * (1 if ws is None else ws[None, :])

    def il_no_deinterleave(x, cos, sin):    # output left interleaved
        r = orig_il(x, cos, sin)
        out = np.empty_like(r)
        h = r.shape[-1] // 2
        out[..., 0::2], out[..., 1::2] = r[..., :h], r[..., h:]
        return out

    def q_half_away(x, sc, of, nax, qtype="int8"):   # rounding half away from zero
        v, pre = orig_q(x, sc, of, nax, qtype)
        if pre is None:
            return v, pre
        return np.clip(np.sign(pre) * np.floor(np.abs(pre) + 0.5), -128, 127).astype(np.int64), pre

    def q_offset_after_round(x, sc, of, nax, qtype="int8"):
        v, pre = orig_q(x, sc, None, nax, qtype)
        if pre is None or of is None:
            return v, pre
        o = np.asarray(of, np.float64)
        o = o[None, :, None, :] if nax else o
        return np.clip(v + np.rint(o), -128, 127).astype(np.int64), pre

    def e4m3_bias8(c):                      # exponent bias 8 instead of 7
        return orig_e4(c) * 0.5

    def kvn_mean_over_all(x, g, eps):       # RMS over the whole last dim + 1
        n = x.shape[-1] + 1
        rms = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) / n + eps)
        return x / rms * g

    orig_enc = orq.encode_e4m3_rne_sat
    orig_rq = orq.row_quantize

    def enc_half_away(v):                   # E4M3 ties rounded away from zero
        v = np.asarray(v, np.float32)
        c = orig_enc(v)
        up = orig_enc(np.nextafter(np.abs(v), np.float32(np.inf)) * np.where(np.signbit(v), -1, 1))
        mags = codes.decode_e4m3(np.arange(127, dtype=np.uint8))
        mids = (mags[:-1] + mags[1:]) / 2
        tie = np.isin(np.abs(v).astype(np.float64), mids)
        return np.where(tie, up, c).astype(np.uint8)

    def enc_no_saturation(v):               # out-of-range magnitudes become NaN codes
        v = np.asarray(v, np.float32)
        c = orig_enc(v)
        return np.where(np.abs(v) > 448, (c & 0x80) | 0x7F, c).astype(np.uint8)

    def rq_fnuz_range(bits):                # scaled onto +-240 instead of +-448
        c, sc = orig_rq(bits)
        x = codes.decode_bf16(np.asarray(bits, np.uint16)).astype(np.float32)
        safe = np.maximum(np.max(np.abs(x), axis=1), np.float32(2.0 ** -100)).astype(np.float32)
        return orig_enc(x * (np.float32(240) / safe)[:, None]), (safe / np.float32(240)).astype(np.float32)

    def rq_reciprocal(bits):                # x times RN(448 / m) in place of x / scale
        c, sc = orig_rq(bits)
        x = codes.decode_bf16(np.asarray(bits, np.uint16)).astype(np.float32)
        safe = np.maximum(np.max(np.abs(x), axis=1), np.float32(2.0 ** -100)).astype(np.float32)
        return orig_enc((x * (np.float32(448) / safe)[:, None]).astype(np.float32)), sc

    orig_slots = okv.token_slots
    orig_rows = okv.cache_rows
    orig_fp8 = codes.encode_fp8

    def slots_blk_per_token(index, mode, b, s, S, bs):   # PA_BLK_BNSD index read per token
        if mode == "PA_BLK_BNSD":
            idx = np.asarray(index, np.int64).reshape(-1)
            return idx[np.minimum(b * S + s, idx.size - 1)]
        return orig_slots(index, mode, b, s, S, bs)

    def rows_norm_ignores_batch(mode, b, p, bs):          # Norm: every batch into batch 0's cache
        return orig_rows(mode, np.zeros_like(b) if mode == "Norm" else b, p, bs)

    def fp8_no_saturation(v, fmt):                       # out-of-range magnitudes become NaN codes
        c = orig_fp8(v, fmt)
        top = 448.0 if fmt == "e4m3" else 57344.0
        return np.where(np.abs(np.asarray(v, np.float64)) > top, (c & 0x80) | 0x7F, c).astype(np.uint8)

    orig_ph = oq.rms_norm_per_head

    def ph_over_all_heads(x, g, eps, d):          # per-head norm taken over the whole segment
        return oq.rms_norm_across_heads(x, np.tile(g, x.shape[1] // d), eps)

    return [(oq, "rms_norm_per_head", ph_over_all_heads), (okv, "token_slots", slots_blk_per_token), (okv, "cache_rows", rows_norm_ignores_batch),
            (codes, "encode_fp8", fp8_no_saturation),
            (orq, "encode_e4m3_rne_sat", enc_half_away), (orq, "encode_e4m3_rne_sat", enc_no_saturation),
            (orq, "row_quantize", rq_fnuz_range), (orq, "row_quantize", rq_reciprocal),
            (oq, "rope_rotate_half", rh_sign), (oq, "rms_norm_across_heads", norm_no_eps),
            (oq, "rms_norm_across_heads", norm_pre_gamma_width), (oq, "dequant_weight", dw_transposed_blocks),
            (okv, "interleave_rope", il_no_deinterleave), (okv, "quantize", q_half_away),
            (okv, "quantize", q_offset_after_round), (codes, "decode_e4m3", e4m3_bias8),
            (okv, "rms_norm", kvn_mean_over_all)]


@pytest.mark.parametrize("i", range(len(mutants())))
def test_mutants(i, monkeypatch):
    mod, name, fn = mutants()[i]
    monkeypatch.setattr(mod, name, fn)
    if mod is codes:  # the code helpers are also bound by name in the oracle modules
        for m in (oq, okv):
            if hasattr(m, name):
                monkeypatch.setattr(m, name, fn)
    caught = []
    for check in ALL_CHECKS:
        try:
            check()
        except (AssertionError, ValueError):
            caught.append(check.__name__)
    assert caught, f"mutant {name}/{fn.__name__} survived every check"


@pytest.mark.parametrize("fmt,tdtype,top", [("e4m3", torch.float8_e4m3fn, 0x7E), ("e5m2", torch.float8_e5m2, 0x7B)])
def test_fp8_neighbours_bracket_the_value(fmt, tdtype, top):
    """The FP8 parity rule's helper: the codes just below and above |v| (v's sign),
    adjacent in code order, with their midpoint; torch's cast and the oracle's
    encoder both land on one of them."""
    decode = {"e4m3": codes.decode_e4m3, "e5m2": codes.decode_e5m2}[fmt]
    mags = decode(np.arange(top + 1, dtype=np.uint8))
    g = np.random.default_rng(11)
    v = np.concatenate([mags, (mags[:-1] + mags[1:]) / 2, g.uniform(0, mags[-1], 4000),
                        np.exp(g.uniform(np.log(mags[1]), np.log(mags[-1]), 4000))])
    v = np.concatenate([v, -v]).astype(np.float32).astype(np.float64)  # values torch can take exactly
    lo, hi, mid = codes.fp8_neighbours(v, fmt)
    mlo, mhi = lo & 0x7F, hi & 0x7F
    assert ((mhi - mlo.astype(np.int64)) <= 1).all() and (mhi >= mlo).all()
    assert (mhi <= top).all()
    a = np.abs(v)
    assert (mags[mlo] <= a).all() and (a <= mags[mhi]).all()
    assert np.array_equal(mid, (mags[mlo] + mags[mhi]) / 2)
    sign = np.signbit(v)
    assert np.array_equal((lo >> 7).astype(bool), sign) and np.array_equal((hi >> 7).astype(bool), sign)
    enc = codes.encode_fp8(v, fmt)
    assert ((enc == lo) | (enc == hi)).all()
    ref = torch.from_numpy(v.astype(np.float32)).to(tdtype).view(torch.uint8).numpy()
    assert ((ref == lo) | (ref == hi)).all()
    # a value on a code comes back as that code's magnitude at the top of the bracket
    on = np.arange(1, top + 1)
    lo_on, hi_on, _ = codes.fp8_neighbours(mags[on], fmt)
    assert np.array_equal(hi_on, on.astype(np.uint8)) and np.array_equal(lo_on, (on - 1).astype(np.uint8))
