"""No kernel writes outside its output tensors.

Every output here is a view into a larger device buffer whose bands before and
after it (4 KB each, so the view keeps the alignment the calls ask for) are
filled with a sentinel.  After the call the bands must still hold the sentinel,
bit for bit, and the output must match the oracle.  The cases take the ragged
edges of each kernel: token counts that are not a multiple of the projection's
256-row pair tile, a column count that is not a multiple of its 256-column tile,
the NBSd layout, the per-head norm, the pipelined norm/RoPE pass (whose bulk
stores write whole spans), the row quantiser's split and packed layouts, and the
KV outputs k_rope / c_kv of the pipelined and register kernels.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import as_f64, check_kv, check_qkv, qkv_reference
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096


class Guarded:
    """`shape` elements of `dtype` between two sentinel bands."""

    def __init__(self, shape, dtype, sentinel: int):
        self.n = int(np.prod(shape))
        bits = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32,
                torch.uint8: torch.uint8, torch.int8: torch.int8}[dtype]
        esz = torch.tensor([], dtype=bits).element_size()
        self.g = GUARD_BYTES // esz
        self.sentinel = sentinel
        self.buf = torch.full((self.n + 2 * self.g,), sentinel, dtype=bits, device="cuda")
        self.view = self.buf[self.g:self.g + self.n].view(dtype).view(shape)

    def check(self, what: str):
        b = self.buf.cpu()
        lo, hi = b[:self.g], b[self.g + self.n:]
        assert bool((lo == self.sentinel).all()), f"{what}: write before the output"
        assert bool((hi == self.sentinel).all()), f"{what}: write after the output"


QKV = [
    # name, make_qkv kwargs, layout
    ("bsd_ragged_rows", dict(S=300, H=256, num_heads=4, num_kv_heads=4, head_dim=64), native.RA_LAYOUT_BSD),
    ("bsd_ragged_cols", dict(S=270, H=256, num_heads=3, num_kv_heads=1, head_dim=64), native.RA_LAYOUT_BSD),
    ("nbsd", dict(S=300, H=256, num_heads=2, num_kv_heads=2, head_dim=128), native.RA_LAYOUT_NBSD),
    ("per_head", dict(S=290, H=256, num_heads=2, num_kv_heads=2, head_dim=128, q_norm="per_head",
                      k_norm="per_head"), native.RA_LAYOUT_BSD),
    ("no_rope_q_only", dict(S=129, H=256, num_heads=4, num_kv_heads=0, head_dim=64, rope=None),
     native.RA_LAYOUT_BSD),
]


@pytest.mark.parametrize("name,kw,layout", QKV, ids=[q[0] for q in QKV])
def test_qkv_output_bands(name, kw, layout):
    case = synth.make_qkv("guard_" + name, 60 + len(name), **kw)
    run = runner.QkvRun(case, layout=layout)
    g = Guarded(tuple(run.out.shape), torch.bfloat16, 0x7FBF)
    run.out = g.view
    run.run()
    torch.cuda.synchronize()
    assert run.status() == 0
    g.check(name)
    got = as_f64(run.out)
    if layout == native.RA_LAYOUT_NBSD:  # [I / d, T, d] -> [T, I]
        got = got.transpose(1, 0, 2).reshape(case.T, case.I)
    check_qkv(case, got, qkv_reference(case), name)


@pytest.mark.parametrize("T,H", [(37, 264), (5, 8200)], ids=["register", "two_pass"])
def test_row_quant_output_bands(T, H):
    bits = synth.hidden_bf16(70 + T, T, H)
    x = runner.to_dev(bits)
    codes = Guarded((T, H), torch.uint8, 0x55)
    scale = Guarded((T,), torch.float32, 0x7FC00001)
    packed = Guarded((T, H + 4), torch.uint8, 0x55)
    native.row_quantize_e4m3(x, codes.view, scale.view)
    native.row_quantize_e4m3_packed(x, packed.view)
    torch.cuda.synchronize()
    for g, what in ((codes, "codes"), (scale, "scale"), (packed, "packed")):
        g.check(what)
    c_ref, s_ref = oracle.row_quantize(bits)
    assert np.array_equal(codes.view.cpu().numpy(), c_ref)
    assert np.array_equal(scale.view.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(packed.view.cpu().numpy(), oracle.row_quantize_packed(bits))


KV = [
    ("v1_pipelined", dict(variant=1, B=2, N=1, S=37, Dkv=576, Dv=512, block_size=32, block_num=4,
                          quant_k=True, quant_v=True)),
    ("v2_pipelined", dict(variant=2, B=2, N=8, S=21, Dkv=192, Dv=128, block_size=32, block_num=2,
                          quant_k=True, quant_v=True)),
    ("v2_register_norm", dict(variant=2, B=2, N=2, S=19, Dkv=192, Dv=128, cache_mode="Norm", cache_seq=24,
                              quant_k=True, quant_v=True)),
    ("v1_register_small", dict(variant=1, B=2, N=1, S=11, Dkv=136, Dv=128, rope_size=8, block_size=16,
                               block_num=2)),
]


@pytest.mark.parametrize("name,kw", KV, ids=[k[0] for k in KV])
def test_kv_output_bands(name, kw):
    case = synth.make_kv("guard_" + name, 80 + len(name), is_output_kv=True, skip_frac=0.1, **kw)
    run = runner.KvRun(case)
    assert run.outputs
    kr = Guarded(tuple(run.k_rope.shape), torch.bfloat16, 0x7FBF)
    ckv = Guarded(tuple(run.c_kv.shape), torch.bfloat16, 0x7FBF)
    run.k_rope, run.c_kv = kr.view, ckv.view
    run.run()
    torch.cuda.synchronize()
    assert native.kv_rms_norm_rope_cache_status() == 0
    kr.check(name + " k_rope")
    ckv.check(name + " c_kv")
    check_kv(case, run, name)


def test_short_cache_is_refused_before_launch():
    """A cache one block short of what the parameters address is refused by the
    binding (the C ABI cannot see buffer sizes), and nothing is launched: the
    caches keep their sentinel."""
    case = synth.make_kv("guard_short", 99, variant=2, B=2, N=8, S=21, Dkv=192, Dv=128, block_size=32,
                         block_num=2, quant_k=True, quant_v=True)
    run = runner.KvRun(case)
    full = run.k_cache
    run.k_cache = full[:-1]
    with pytest.raises(ValueError, match=r"^k_cache: the call needs"):
        run.run()
    torch.cuda.synchronize()
    assert np.array_equal(full.cpu().numpy(), case.k_cache)
    assert np.array_equal(run.ckv_cache.cpu().numpy(), case.ckv_cache)
