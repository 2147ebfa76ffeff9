"""Failure detection in the projection and KV cache pipelines, without a GPU fault.

Every wait in the projection kernel's pipeline (TMA stage barriers, the
accumulator hand-over between the MMA issuer and the epilogue) has a time
limit.  The test hook ra_test_stall_next_projection makes the next launch issue
none of its loads, so its waits run out with nothing in flight.  The kernel must
record the timeout in the workspace status word (read on the host through
qkv_cte_mx_status, which also clears it), release its tensor memory and exit;
the CUDA context must stay usable, and the next call, with the hook cleared,
must give the correct result.  The pipelined norm/RoPE pass (through
ra_test_stall_next_norm_rope and the same status word) and the pipelined KV
cache kernel (through ra_test_stall_next_kv_cache and
kv_rms_norm_rope_cache_status) are held to the same rules.
"""
import ctypes

import pytest
import torch

from parity_util import as_f64, check_kv, check_qkv, qkv_reference
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu

DEFAULT_WAIT_NS = 2_000_000_000


def test_stalled_pipeline_reports_timeout_and_context_survives():
    case = synth.qkv_tiny()
    run = runner.QkvRun(case)
    native.ra_set_wait_timeout_ns(2_000_000)  # 2 ms per wait
    try:
        native.ra_test_stall_next_projection()
        run.project()
        # the status word is set by every CTA that gave up; the C entry point reports it
        v = ctypes.c_int32()
        st = native.load().qkv_cte_mx_status(ctypes.c_void_p(run.workspace.data_ptr()), None,
                                             ctypes.byref(v))
        assert st == -6 and v.value == 1, (st, v.value)
        assert "ran out of time" in native.load().ra_last_error().decode()
        # the word was cleared by the read, and the hook applied to one launch only
        run.run()
        torch.cuda.synchronize()
        assert run.status() == 0
    finally:
        native.ra_set_wait_timeout_ns(DEFAULT_WAIT_NS)
    check_qkv(case, as_f64(run.out), qkv_reference(case), "call after a timed-out launch")


@pytest.mark.parametrize("layout", [native.RA_LAYOUT_BSD, native.RA_LAYOUT_NBSD], ids=["bsd", "nbsd"])
def test_stalled_norm_rope_pipeline_reports_timeout_and_context_survives(layout):
    case = synth.qkv_tiny()
    run = runner.QkvRun(case, layout=layout)
    native.ra_set_wait_timeout_ns(2_000_000)  # 2 ms per wait
    try:
        run.project()
        torch.cuda.synchronize()
        assert run.status() == 0
        native.ra_test_stall_next_norm_rope()
        run.norm_rope()
        v = ctypes.c_int32()
        st = native.load().qkv_cte_mx_status(ctypes.c_void_p(run.workspace.data_ptr()), None,
                                             ctypes.byref(v))
        assert st == -6 and v.value == 1, (st, v.value)
        # cleared by the read; the hook applied to one launch only
        run.run()
        torch.cuda.synchronize()
        assert run.status() == 0
    finally:
        native.ra_set_wait_timeout_ns(DEFAULT_WAIT_NS)
    out = run.out
    if layout == native.RA_LAYOUT_NBSD:  # [I / d, T, d] -> [T, I]
        out = out.permute(1, 0, 2).reshape(case.T, case.I)
    check_qkv(case, as_f64(out), qkv_reference(case), "call after a timed-out norm/RoPE pass")


def test_stalled_kv_pipeline_reports_timeout_and_context_survives():
    # V2 with the common row shape, PA_BNSD, int8: the pipelined kernel
    case = synth.make_kv("stall_kv", 11, variant=2, B=2, N=8, S=40, Dkv=192, Dv=128, block_size=32,
                         block_num=4, quant_k=True, quant_v=True)
    native.ra_set_wait_timeout_ns(2_000_000)  # 2 ms per wait
    try:
        assert native.kv_rms_norm_rope_cache_status() == 0
        native.ra_test_stall_next_kv_cache()
        runner.KvRun(case).run()
        v = ctypes.c_int32()
        st = native.load().kv_rms_norm_rope_cache_status(None, ctypes.byref(v))
        assert st == -6 and v.value == 1, (st, v.value)
        assert "ran out of time" in native.load().ra_last_error().decode()
        # cleared by the read; the hook applied to one call only
        run = runner.KvRun(case)
        run.run()
        torch.cuda.synchronize()
        assert native.kv_rms_norm_rope_cache_status() == 0
    finally:
        native.ra_set_wait_timeout_ns(DEFAULT_WAIT_NS)
    check_kv(case, run, "call after a timed-out launch")
