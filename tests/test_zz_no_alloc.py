"""qkv_cte_mx_noalloc: the prologue for callers that cannot allocate device memory.

Some host programs must not call cudaMalloc where they run this operator (a
plugin of an inference runtime that owns all device memory, or a serving loop
that cannot take cudaMalloc's implicit device synchronisation).  For them the
library keeps its scratch in a static device array and the entry point takes
no workspace.  These tests call it through the C ABI and check it against the
regular entry point (caller-owned workspace) with the parity tolerance, on two
calls in a row, and check that oversized problems are refused before launch.
This file sorts last so a failure here stops a -x run only after every other
test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import as_f64, check_qkv
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu


def _noalloc(run, out):
    native.qkv_cte_mx_noalloc(run.params, run.a, run.a_scale, run.w_packed, run.weight_scales,
                              run.bias, run.cos, run.sin, run.q_gamma, run.k_gamma, out)


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
    expected = as_f64(run.out)
    for call in range(2):  # the static array keeps the previous call's contents
        out = torch.full_like(run.out, float("nan"))
        _noalloc(run, out)
        torch.cuda.synchronize()
        check_qkv(case, as_f64(out), expected, f"noalloc call {call}")


def test_noalloc_rejects_oversized_problem():
    lib = native.load()
    p = native.QkvCteMxParams(B=4, S=1 << 20, H=5120, num_heads=40, num_kv_heads=40, head_dim=128,
                              q_norm=1, k_norm=1, fused_rope=1, norm_eps=1e-6, output_layout=0)
    # the call below passes placeholder addresses: it must be refused before any launch,
    # so make sure the problem really needs more scratch than the static array holds
    need = ctypes.c_size_t()
    assert lib.qkv_cte_mx_workspace_bytes(ctypes.byref(p), ctypes.byref(need)) == 0
    assert need.value > 4 * (32 << 20)
    a16 = 0x10000  # never dereferenced
    st = lib.qkv_cte_mx_noalloc(ctypes.byref(p), a16, a16, a16, None, a16, a16, a16, a16, a16, a16, None)
    assert st == -4
    assert "static workspace" in lib.ra_last_error().decode()
