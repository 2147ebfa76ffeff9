"""Plain fp64 CPU oracle for the attention prologue -- TEST INFRASTRUCTURE ONLY.

This package is the independent reference that the CUDA path is checked
against.  It is slow on purpose: numpy in float64, whole-array steps in the
order the pages give them, no blocking, fusion or reordering.  It shares no
code with the CUDA path and never imports it.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may import it.  The product
path (``rope_attention_gb300``'s binding and the C-ABI library) never calls
into it and has no CPU fallback.

Modules
-------
codes     : decoding of e4m3 / ue8m0 / bf16 codes (OCP FP8 and bfloat16 formats).
qkv_cte   : fused QKV projection + across-heads RMSNorm + rotate-half RoPE
            (AWS Neuron "Kernel reference: qkv_cte", Pattern, Upstream behavior,
            Design 1a-1c, Design 2, Design 5).
kv_cache  : KvRmsNormRopeCache (CANN ops-transformer "KvRmsNormRopeCache",
            formulas (1)-(5)).
row_quant : row FP8 quantisation of the activation into the row-packed layout
            (AWS Neuron "Kernel reference: qkv_cte", Interface).

Every function is pinned by ``tests/test_oracle_pins.py``; no function here is
"parity unpinned".
"""
from .codes import decode_bf16, decode_e4m3, decode_ue8m0  # noqa: F401
from .kv_cache import kv_rms_norm_rope_cache  # noqa: F401
from .qkv_cte import qkv_cte_mx  # noqa: F401
from .row_quant import row_quantize, row_quantize_packed  # noqa: F401
