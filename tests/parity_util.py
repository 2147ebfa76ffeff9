"""Comparison rules shared by the GPU parity tests.

Tolerances (the tolerance this project's numerics target states):
* bf16 outputs: |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref row), where the row is
  the token's vector in that output (for the projection: its Q, K or V segment);
* scatter placement and untouched cache slots: bit-exact;
* int8 cache codes: equal, except +-1 where the oracle's pre-rounding value lies
  within 1e-3 of a .5 tie.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def check_bf16(got: np.ndarray, ref: np.ndarray, what: str, rtol: float = 1e-2, row_tol: float = 1e-2):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    tol = rtol * np.abs(ref) + row_tol * rms
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err / np.maximum(tol, 1e-300), 0)), bad.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {idx}: "
            f"gpu={got[idx]!r} ref={ref[idx]!r} tol={tol[idx]!r}")
    return float(np.max(err / np.maximum(tol, 1e-300))) if err.size else 0.0


def check_int8(got: np.ndarray, ref: np.ndarray, pre: np.ndarray, what: str) -> int:
    """Returns the number of +-1 differences at ties."""
    got = np.asarray(got, np.int64)
    ref = np.asarray(ref, np.int64)
    diff = got - ref
    tie = np.abs(pre - (np.floor(pre) + 0.5)) <= 1e-3
    ok = (diff == 0) | ((np.abs(diff) == 1) & tie)
    if not ok.all():
        idx = np.unravel_index(np.argmin(ok), ok.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} int8 codes differ; first at {idx}: "
                             f"gpu={got[idx]} ref={ref[idx]} pre={pre[idx]!r}")
    return int(np.count_nonzero(diff))


def check_fp8(got: np.ndarray, ref: np.ndarray, pre: np.ndarray, fmt: str, what: str) -> int:
    """FP8 cache codes: equal to the oracle's, or the other neighbour of the oracle's
    pre-rounding value when that value lies within 1e-3 (relative) of the midpoint
    between the two (the kernel rounds an fp32 value, the oracle an fp64 one).
    Returns the number of such differences."""
    got = np.asarray(got, np.int64)
    ref = np.asarray(ref, np.int64)
    lo, hi, mid = oracle.codes.fp8_neighbours(pre, fmt)
    near_tie = np.abs(np.abs(pre) - mid) <= 1e-3 * np.maximum(mid, 1e-30)
    other = np.where(ref == lo.astype(np.int64), hi.astype(np.int64), lo.astype(np.int64))
    ok = (got == ref) | ((got == other) & near_tie)
    if not ok.all():
        idx = np.argmin(ok)
        raise AssertionError(f"{what}: {int((~ok).sum())} {fmt} codes differ; first: gpu={got.ravel()[idx]:#x} "
                             f"ref={ref.ravel()[idx]:#x} pre={pre.ravel()[idx]!r}")
    return int(np.count_nonzero(got != ref))


def qkv_reference(case, rows: np.ndarray | None = None) -> np.ndarray:
    c = case
    sel = slice(None) if rows is None else rows
    return oracle.qkv_cte_mx(
        c.a[sel], c.a_scale[sel], c.w, c.w_block_exp, num_heads=c.num_heads,
        num_kv_heads=c.num_kv_heads, head_dim=c.head_dim, weight_scales=c.weight_scales,
        bias=c.bias, q_norm=c.q_norm, k_norm=c.k_norm, q_gamma=c.q_gamma, k_gamma=c.k_gamma,
        eps=c.eps, fused_rope=c.fused_rope, cos=None if c.cos is None else c.cos[sel],
        sin=None if c.sin is None else c.sin[sel])


def check_qkv(case, got: np.ndarray, ref: np.ndarray, what: str) -> float:
    qw = case.num_heads * case.head_dim
    kw = case.num_kv_heads * case.head_dim
    worst = check_bf16(got[:, :qw], ref[:, :qw], f"{what} Q")
    if kw:
        worst = max(worst, check_bf16(got[:, qw:qw + kw], ref[:, qw:qw + kw], f"{what} K"))
        worst = max(worst, check_bf16(got[:, qw + kw:], ref[:, qw + kw:], f"{what} V"))
    return worst


def kv_reference(case) -> dict:
    c = case
    return oracle.kv_rms_norm_rope_cache(
        c.kv, c.gamma, c.cos, c.sin, c.index, c.k_cache, c.ckv_cache, variant=c.variant,
        rope_size=c.rope_size, block_size=c.block_size, cache_mode=c.cache_mode, epsilon=c.eps,
        k_scale=c.k_scale, k_offset=c.k_offset, v_scale=c.v_scale, v_offset=c.v_offset, v=c.v,
        is_output_kv=c.is_output_kv, dtype=c.dtype, k_qtype=c.k_qtype, v_qtype=c.v_qtype)


def check_kv(case, run, what: str) -> dict:
    """Compare every output of a KvRun against the oracle; returns mismatch statistics."""
    ref = kv_reference(case)
    stats = {}
    for name, init, quant, qtype in (("k_cache", case.k_cache, case.k_scale is not None, case.k_qtype),
                                     ("ckv_cache", case.ckv_cache, case.v_scale is not None, case.v_qtype)):
        dev = getattr(run, name)
        written = ref["k_written" if name == "k_cache" else "ckv_written"]
        if quant:
            got = dev.cpu().numpy().astype(np.int64)
            untouched_ok = np.array_equal(got[~written], init.astype(np.int64)[~written])
            assert untouched_ok, f"{what} {name}: a slot outside the index map was modified"
            pre = ref["k_pre" if name == "k_cache" else "ckv_pre"]
            if qtype == "int8":
                stats[name + "_ties"] = check_int8(got[written], ref[name][written], pre[written], f"{what} {name}")
            else:
                stats[name + "_ties"] = check_fp8(got[written], ref[name][written], pre[written], qtype,
                                                  f"{what} {name}")
        else:
            bits = dev.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(bits[~written], init[~written]), \
                f"{what} {name}: a slot outside the index map was modified"
            got = as_f64(dev)
            rows_w = written.all(axis=-1)
            assert np.array_equal(rows_w, written.any(axis=-1)), f"{what} {name}: partial row write"
            check_bf16(got[rows_w], ref[name][rows_w], f"{what} {name}")
    assert run.outputs == ("k_rope" in ref), f"{what}: the outputs' on/off rule differs from the oracle"
    if run.outputs:
        check_bf16(as_f64(run.k_rope), ref["k_rope"], f"{what} k_rope")
        check_bf16(as_f64(run.c_kv), ref["c_kv"], f"{what} c_kv")
    assert int(run.err.item()) == ref["bad_index"], f"{what}: bad-index count {run.err.item()} != {ref['bad_index']}"
    return stats
