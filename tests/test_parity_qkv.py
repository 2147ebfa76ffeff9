"""GPU parity: qkv_cte_mx (C-ABI) against the fp64 oracle.

Small cases are compared in full: they span several 256 x 256 pair tiles,
ragged row and column tails, single-segment calls, per-channel weight
scales, no bias, norm without RoPE and RoPE without norm.  The full-size Wan
workloads are compared on a deterministic row sample (first 128 rows, last
256 rows covering the M tail, 640 random rows) with every column, so the
across-heads norms are checked exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import as_f64, check_bf16, check_qkv, qkv_reference
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu


def run_full(case, split=False, layout=native.RA_LAYOUT_BSD):
    r = runner.QkvRun(case, layout=layout)
    if split:
        r.project()
        r.norm_rope()
    else:
        r.run()
    torch.cuda.synchronize()
    assert r.status() == 0
    return r


def test_tiny_config():
    """S=128, H=256, n_q=n_kv=2, d=64, 1-D RoPE (the small self-attention workload)."""
    case = synth.qkv_tiny()
    r = run_full(case)
    check_qkv(case, as_f64(r.out), qkv_reference(case), "tiny")


SMALL = [
    ("ragged_rows_cols", dict(S=333, H=384, num_heads=3, num_kv_heads=1, head_dim=64)),
    ("batch2_ragged", dict(B=2, S=100, H=256, num_heads=2, num_kv_heads=2, head_dim=128)),
    ("weight_scales_nobias", dict(S=256, H=512, num_heads=4, num_kv_heads=2, head_dim=64,
                                  weight_scales=True, bias=False)),
    ("norm_no_rope", dict(S=200, H=256, num_heads=4, num_kv_heads=4, head_dim=64, rope=None)),
    ("rope_no_norm", dict(S=130, H=256, num_heads=2, num_kv_heads=2, head_dim=64,
                          q_norm=False, k_norm=False)),
    ("q_norm_only", dict(S=129, H=256, num_heads=2, num_kv_heads=2, head_dim=64, k_norm=False)),
    ("single_segment_q", dict(S=300, H=512, num_heads=6, num_kv_heads=0, head_dim=128, rope=None)),
    ("single_segment_v", dict(S=77, H=256, num_heads=2, num_kv_heads=0, head_dim=128, rope=None,
                              q_norm=False)),
    ("one_row", dict(S=1, H=128, num_heads=1, num_kv_heads=1, head_dim=16)),
    ("wide_heads", dict(S=260, H=640, num_heads=5, num_kv_heads=5, head_dim=128)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
def test_small(name, kw):
    case = synth.make_qkv(name, 200 + len(name), **kw)
    r = run_full(case)
    check_qkv(case, as_f64(r.out), qkv_reference(case), name)


# The projection's MMA issuer takes one of two loops by the number of 128-deep K steps
# (H / 128): an even count issues two pipeline stages per asm block with a look-ahead
# probe of the next pair's full barriers, an odd count one stage per bounded wait.
# 2600 rows x 2048 columns are 88 pair tiles, more than there are CTA pairs, so some
# pairs run two tiles and carry the ring position and the look-ahead across a tile.
K_STEPS = [1, 2, 3, 6, 7, 12]


@pytest.mark.parametrize("k_steps", K_STEPS, ids=[f"k_steps_{k}" for k in K_STEPS])
def test_mma_issue_paths(k_steps):
    case = synth.make_qkv(f"k_steps_{k_steps}", 300 + k_steps, S=2600, H=128 * k_steps, num_heads=8,
                          num_kv_heads=4, head_dim=128)
    r = run_full(case)
    check_qkv(case, as_f64(r.out), qkv_reference(case), case.name)


NBSD = [
    ("tiny_qkv", dict(S=128, H=256, num_heads=2, num_kv_heads=2, head_dim=64)),
    ("batch2_ragged", dict(B=2, S=100, H=256, num_heads=2, num_kv_heads=2, head_dim=128)),
    ("cross_q", dict(S=300, H=512, num_heads=6, num_kv_heads=0, head_dim=128, rope=None)),
    ("cross_v", dict(S=77, H=256, num_heads=2, num_kv_heads=0, head_dim=128, rope=None, q_norm=False)),
    ("d16_one_row", dict(S=1, H=128, num_heads=1, num_kv_heads=1, head_dim=16)),
    # the pipelined NBSd pass: 19 rewritten heads (a full box of 16 and a clipped one)
    # with 7 V planes after them that must stay as projected, and token counts that are
    # not a multiple of the tokens per stage
    ("heads19_d128", dict(S=1001, H=256, num_heads=12, num_kv_heads=7, head_dim=128)),
    ("heads19_d64", dict(B=3, S=333, H=256, num_heads=12, num_kv_heads=7, head_dim=64)),
    ("heads33_norm_only_d64", dict(S=517, H=256, num_heads=20, num_kv_heads=13, head_dim=64, rope=None)),
    ("q_norm_only_d128", dict(S=259, H=256, num_heads=5, num_kv_heads=3, head_dim=128, k_norm=False)),
    ("two_rows", dict(S=2, H=128, num_heads=3, num_kv_heads=2, head_dim=64)),
]


@pytest.mark.parametrize("name,kw", NBSD, ids=[s[0] for s in NBSD])
@pytest.mark.parametrize("split", [False, True], ids=["fused", "split"])
def test_nbsd_layout(name, kw, split):
    """output_layout NBSd: out [I/d, B, S, d].  The result, read back into [T, I]
    order, passes parity and equals the BSD run bit for bit (same arithmetic); the
    read-back is checked to invert the oracle's NBSd layout map."""
    case = synth.make_qkv(name, 300 + len(name), **kw)
    T, I, d = case.T, case.I, case.head_dim
    r = run_full(case, split=split, layout=native.RA_LAYOUT_NBSD)
    g = r.out.view(torch.int16).cpu().numpy()               # [n, T, d] bf16 bits
    back = g.transpose(1, 0, 2).reshape(T, I)                 # -> [T, I]
    assert np.array_equal(oracle.qkv_cte.to_nbsd(back, case.B, case.S, d).reshape(g.shape), g)
    bsd = run_full(case, split=split)
    assert np.array_equal(back, bsd.out.view(torch.int16).cpu().numpy()), "NBSd != BSD"
    check_qkv(case, as_f64(torch.from_numpy(back).view(torch.bfloat16)), qkv_reference(case), name)


PER_HEAD = [
    ("ph128_rope", dict(S=260, H=512, num_heads=4, num_kv_heads=4, head_dim=128, q_norm="per_head",
                        k_norm="per_head")),
    ("ph64_odd_heads", dict(S=333, H=384, num_heads=3, num_kv_heads=1, head_dim=64, q_norm="per_head",
                            k_norm="per_head")),
    ("ph_q_across_k", dict(S=200, H=256, num_heads=3, num_kv_heads=2, head_dim=64, q_norm="per_head")),
    ("across_q_ph_k", dict(S=129, H=256, num_heads=2, num_kv_heads=2, head_dim=128, k_norm="per_head")),
    ("ph_no_rope", dict(S=150, H=256, num_heads=2, num_kv_heads=2, head_dim=128, q_norm="per_head",
                        k_norm="per_head", rope=None)),
    ("ph_q_only_segment", dict(S=100, H=256, num_heads=4, num_kv_heads=0, head_dim=64, q_norm="per_head")),
]


@pytest.mark.parametrize("name,kw", PER_HEAD, ids=[s[0] for s in PER_HEAD])
def test_per_head_norm(name, kw):
    """The upstream per-head qk-norm (+ RoPE), finished in the projection epilogue."""
    case = synth.make_qkv(name, 500 + len(name), **kw)
    r = run_full(case)
    check_qkv(case, as_f64(r.out), qkv_reference(case), name)
    s = run_full(case, split=True)
    assert torch.equal(r.out.view(torch.int16), s.out.view(torch.int16)), "split != fused"


def test_per_head_norm_nbsd():
    case = synth.make_qkv("ph_nbsd", 77, B=2, S=90, H=256, num_heads=2, num_kv_heads=2, head_dim=128,
                          q_norm="per_head", k_norm="per_head")
    r = run_full(case, layout=native.RA_LAYOUT_NBSD)
    g = r.out.view(torch.int16).cpu().numpy()
    back = g.transpose(1, 0, 2).reshape(case.T, case.I)
    check_qkv(case, as_f64(torch.from_numpy(back).view(torch.bfloat16)), qkv_reference(case), "ph_nbsd")


def test_output_only_16_byte_aligned():
    """The epilogue writes 32-byte pieces when `out` is 32-byte aligned and 16-byte
    pieces otherwise: an `out` that starts 16 bytes into a buffer takes the second
    path and must give the same bits."""
    case = synth.make_qkv("align16", 12, S=200, H=256, num_heads=2, num_kv_heads=2, head_dim=64)
    a = run_full(case)
    b = runner.QkvRun(case)
    buf = torch.empty(case.T * case.I + 64, dtype=torch.bfloat16, device="cuda")
    b.out = buf[8:8 + case.T * case.I].view(case.T, case.I)  # 16 bytes past a 32-byte boundary
    assert b.out.data_ptr() % 32 == 16
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_split_entry_points_match_fused():
    case = synth.make_qkv("split", 5, S=250, H=256, num_heads=3, num_kv_heads=3, head_dim=64)
    a = run_full(case)
    b = run_full(case, split=True)
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_deterministic():
    case = synth.make_qkv("det", 6, S=500, H=512, num_heads=4, num_kv_heads=4, head_dim=128)
    r = run_full(case)
    first = r.out.clone()
    r.run()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), r.out.view(torch.int16))


def test_projection_only_matches_oracle_projection():
    """With norms and RoPE off, qkv_cte_mx_project is the whole operator."""
    case = synth.make_qkv("proj", 7, S=389, H=1024, num_heads=4, num_kv_heads=4, head_dim=128,
                          rope=None, q_norm=False, k_norm=False, weight_scales=True)
    r = runner.QkvRun(case)
    r.project()
    torch.cuda.synchronize()
    ref = qkv_reference(case)
    check_bf16(as_f64(r.out), ref, "projection")


def _sampled(case, what):
    r = run_full(case)
    rows = synth.sample_rows(case.T, seed=123)
    got = as_f64(r.out[torch.from_numpy(rows).cuda()])
    del r
    torch.cuda.empty_cache()
    return check_qkv(case, got, qkv_reference(case, rows), what)


def test_wan480_self_attention_sampled():
    """S=32760 (21x30x52), H=5120, 40+40+40 heads of 128, 3-D RoPE."""
    _sampled(synth.qkv_wan480(), "wan480")


def test_wan_cross_attention_sampled():
    """Separate Q (S=32760, normed), K (L=512, normed) and V (L=512) projections, no RoPE."""
    for case in synth.qkv_wan_cross():
        _sampled(case, case.name)


def test_wan720_self_attention_sampled():
    """S=75600 (21x45x80), the bench workload."""
    _sampled(synth.qkv_wan720(), "wan720")


def test_wan480_nbsd_sampled():
    """The 480p self-attention call with output layout NBSd [120, 1, 32760, 128]: sampled
    rows read back from the 120 head planes, against the oracle."""
    case = synth.qkv_wan480()
    r = run_full(case, layout=native.RA_LAYOUT_NBSD)
    rows = torch.from_numpy(synth.sample_rows(case.T, seed=124)).cuda()
    n = case.I // case.head_dim
    got = r.out.view(n, case.T, case.head_dim)[:, rows, :].permute(1, 0, 2).reshape(len(rows), case.I)
    got = as_f64(got)
    del r
    torch.cuda.empty_cache()
    check_qkv(case, got, qkv_reference(case, rows.cpu().numpy()), "wan480_nbsd")


def _degenerate(case, bias_on: bool):
    """Rows and weight blocks at the edges of what the operator meets: all-zero rows
    (v = bias), rows whose dequant scale is 1e-20 and 1e-30 of the others (v is bias,
    or tiny when there is no bias, so eps dominates their RMS), rows scaled up 1e3, and
    W blocks whose MX exponents are moved 20 binades up or down (columns of one row
    that differ by 2^40, inside the same 128-column blocks of the intermediate)."""
    c = case
    c.a[0:8] = 0
    c.a_scale[8:16] *= np.float32(1e-20)
    c.a_scale[16:24] *= np.float32(1e-30)
    c.a_scale[24:32] *= np.float32(1e3)
    e = c.w_block_exp.astype(np.int32)
    e[1, 0:96] += 20
    e[3, 200:330] -= 20
    c.w_block_exp[:] = np.clip(e, 1, 254).astype(np.uint8)
    return c


@pytest.mark.parametrize("bias", [True, False], ids=["bias", "no_bias"])
def test_degenerate_rows_and_blocks(bias):
    case = _degenerate(synth.make_qkv("degenerate", 71, S=260, H=256, num_heads=3, num_kv_heads=2,
                                      head_dim=64, bias=bias), bias)
    r = run_full(case)
    check_qkv(case, as_f64(r.out), qkv_reference(case), f"degenerate ({'bias' if bias else 'no bias'})")
    s = run_full(case, split=True, layout=native.RA_LAYOUT_NBSD)
    back = s.out.view(torch.int16).cpu().numpy().transpose(1, 0, 2).reshape(case.T, case.I)
    assert np.array_equal(back, r.out.view(torch.int16).cpu().numpy()), "NBSd != BSD"
