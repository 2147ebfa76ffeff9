"""qkv_cte_mx_noalloc: the prologue for callers that cannot allocate device memory.

Some host programs must not call cudaMalloc where they run this operator (a
plugin of an inference runtime that owns all device memory, or a serving loop
that cannot take cudaMalloc's implicit device synchronisation).  For them the
library keeps its scratch in a static device array and the entry point takes
no workspace.  These tests call it through the C ABI and check, on two calls in
a row (the array keeps the previous call's contents), that its output equals
the regular entry point's (caller-owned workspace) bit for bit -- both run the
same kernels on the same inputs -- and matches the oracle within the parity
tolerance; that a pipeline timeout in such a call can be read back; and that
an oversized problem is refused before anything reaches the device.  This file
sorts last so a failure here stops a -x run only after every other test has run.
"""
import ctypes

import pytest
import torch

from parity_util import as_f64, check_qkv, qkv_reference
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu

DEFAULT_WAIT_NS = 2_000_000_000


def _noalloc(run, out):
    native.qkv_cte_mx_noalloc(run.params, run.a, run.a_scale, run.w_packed, run.weight_scales,
                              run.bias, run.cos, run.sin, run.q_gamma, run.k_gamma, out)


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16).cpu()


@pytest.mark.parametrize("kw", [
    dict(S=128, H=256, num_heads=2, num_kv_heads=2, head_dim=64),            # the tiny self-attention shape
    dict(S=333, H=384, num_heads=3, num_kv_heads=1, head_dim=64),            # ragged rows and columns
    dict(S=300, H=512, num_heads=6, num_kv_heads=0, head_dim=128, rope=None),  # single-segment call
], ids=["tiny", "ragged", "single_segment"])
def test_noalloc_matches_workspace_entry_point(kw):
    case = synth.make_qkv("noalloc", 31, **kw)
    run = runner.QkvRun(case)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    expected = _bits(run.out)
    ref = qkv_reference(case)
    for call in range(2):  # the static array keeps the previous call's contents
        out = torch.full_like(run.out, float("nan"))
        _noalloc(run, out)
        torch.cuda.synchronize()
        assert native.qkv_cte_mx_status(None) == 0, f"noalloc call {call}: a pipeline wait ran out"
        got = _bits(out)
        assert torch.equal(got, expected), \
            f"noalloc call {call}: {int((got != expected).sum())} elements differ from qkv_cte_mx"
        check_qkv(case, as_f64(out), ref, f"noalloc call {call}")


def test_noalloc_timeout_is_reported_and_the_next_call_is_exact():
    """A stalled projection launch inside a noalloc call leaves its mark in the static
    array's status word, which qkv_cte_mx_status reads (and clears) when given no
    workspace; the next noalloc call is correct."""
    case = synth.qkv_tiny()
    run = runner.QkvRun(case)
    run.run()
    torch.cuda.synchronize()
    expected = _bits(run.out)
    out = torch.full_like(run.out, float("nan"))
    native.ra_set_wait_timeout_ns(2_000_000)  # 2 ms per wait
    try:
        native.ra_test_stall_next_projection()
        _noalloc(run, out)
        v = ctypes.c_int32()
        st = native.load().qkv_cte_mx_status(None, None, ctypes.byref(v))
        assert st == -6 and v.value == 1, (st, v.value)
        assert "ran out of time" in native.load().ra_last_error().decode()
        _noalloc(run, out)
        torch.cuda.synchronize()
        assert native.qkv_cte_mx_status(None) == 0
    finally:
        native.ra_set_wait_timeout_ns(DEFAULT_WAIT_NS)
    assert torch.equal(_bits(out), expected)


def test_noalloc_rejects_oversized_problem():
    """A problem whose scratch exceeds the static array is refused.  The call passes
    no buffers at all (NULL pointers) with the validate-only hook set, so even a
    regression in the size check could not send anything to the device."""
    lib = native.load()
    p = native.QkvCteMxParams(B=4, S=1 << 20, H=5120, num_heads=40, num_kv_heads=40, head_dim=128,
                              q_norm=1, k_norm=1, fused_rope=1, norm_eps=1e-6, output_layout=0)
    need = ctypes.c_size_t()
    assert lib.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(need)) == 0
    assert need.value > 32 << 20
    lib.ra_test_validate_only(1)
    try:
        st = lib.qkv_cte_mx_noalloc(ctypes.byref(p), None, None, None, None, None, None, None, None, None,
                                    None, None)
    finally:
        lib.ra_test_validate_only(0)
    assert st == -4
    assert "static workspace" in lib.ra_last_error().decode()
