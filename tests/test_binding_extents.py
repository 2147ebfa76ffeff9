"""The binding's size checks, on the CPU (no kernel is launched).

The C ABI takes bare device pointers, so it cannot tell a buffer that is too
short from one that fits; the Python binding refuses a tensor that spans fewer
bytes than the call reads or writes through it.  These tests pin the extents it
computes from the call's parameters against the exact array sizes of seeded
cases in every cache mode, cache type, row shape and optional-argument
combination, and check that a short tensor is refused before anything reaches
the device (the size check runs before the placement check, so CPU tensors
show it).
"""
import pytest
import torch

from rope_attention_gb300 import build, native, runner, synth


@pytest.fixture(scope="module", autouse=True)
def _library():
    """The wrappers reach the library (load()) before they marshal tensors: build it
    if this file runs first in a fresh checkout."""
    build.build()

QKV_CASES = [
    dict(S=16, H=128, num_heads=2, num_kv_heads=2, head_dim=64),
    dict(B=2, S=9, H=256, num_heads=3, num_kv_heads=1, head_dim=128, weight_scales=True, bias=False),
    dict(S=8, H=128, num_heads=4, num_kv_heads=0, head_dim=64, rope=None),
    dict(S=8, H=128, num_heads=2, num_kv_heads=0, head_dim=128, rope=None, q_norm=False),
    dict(S=8, H=128, num_heads=2, num_kv_heads=2, head_dim=64, q_norm="per_head", k_norm="per_head"),
    dict(S=8, H=128, num_heads=2, num_kv_heads=2, head_dim=64, q_norm=False, k_norm=False),
    dict(S=8, H=128, num_heads=2, num_kv_heads=2, head_dim=64, k_norm=False, rope=None),
]


@pytest.mark.parametrize("kw", QKV_CASES, ids=[f"qkv{i}" for i in range(len(QKV_CASES))])
def test_qkv_extents_match_case_arrays(kw):
    c = synth.make_qkv("extents", 7, **kw)
    ext = native.qkv_extents(runner.qkv_params(c))
    assert ext["a"] == c.a.nbytes
    assert ext["a_scale"] == c.a_scale.nbytes
    assert ext["out"] == c.T * c.I * 2
    for name, arr in (("weight_scales", c.weight_scales), ("bias", c.bias), ("q_gamma", c.q_gamma),
                      ("k_gamma", c.k_gamma), ("cos_cache", c.cos), ("sin_cache", c.sin)):
        if arr is not None:
            assert ext[name] == arr.nbytes, name
    if not c.fused_rope:
        assert ext["cos_cache"] == ext["sin_cache"] == 0
    if not c.q_norm:
        assert ext["q_gamma"] == 0
    if not c.k_norm:
        assert ext["k_gamma"] == 0


KV_CASES = [
    dict(variant=1, B=2, N=1, S=37, Dkv=576, Dv=512, block_size=16, block_num=8),
    dict(variant=1, B=2, N=1, S=20, Dkv=576, Dv=512, block_size=32, block_num=2, cache_mode="PA",
         quant_k=True, quant_v=True),
    dict(variant=1, B=2, N=1, S=20, Dkv=576, Dv=512, block_size=32, block_num=2, quant_k=True,
         quant_v=True, k_scalar=True, v_scalar=True),
    dict(variant=1, B=2, N=1, S=20, Dkv=576, Dv=512, block_size=32, cache_mode="Norm", cache_seq=40),
    dict(variant=2, B=2, N=8, S=29, Dkv=192, Dv=128, block_size=32, block_num=4, quant_k=True,
         quant_v=True),
    dict(variant=2, B=3, N=4, S=21, Dkv=192, Dv=128, block_size=16, block_num=8, cache_mode="PA"),
    dict(variant=2, B=2, N=2, S=70, Dkv=192, Dv=128, block_size=32, cache_mode="PA_BLK_BNSD",
         quant_k=True, quant_v=True),
    dict(variant=2, B=2, N=2, S=30, Dkv=192, Dv=128, block_size=32, cache_mode="Norm", cache_seq=48,
         quant_k=True, quant_v=True, k_qtype="e4m3", v_qtype="e5m2"),
    dict(variant=2, B=2, N=2, S=30, Dkv=192, Dv=128, block_size=32, block_num=2, rope_broadcast=True,
         dtype="fp16"),
    dict(variant=2, B=1, N=1, S=13, Dkv=64, Dv=512, rope_size=32, block_size=32, block_num=1,
         quant_v=True, is_output_kv=False),
]


@pytest.mark.parametrize("kw", KV_CASES, ids=[f"kv{i}" for i in range(len(KV_CASES))])
def test_kv_extents_match_case_arrays(kw):
    c = synth.make_kv("extents", 8, **kw)
    ext = native.kv_extents(runner.kv_params(c))
    for name, arr in (("kv", c.kv), ("gamma", c.gamma), ("cos", c.cos), ("sin", c.sin), ("index", c.index),
                      ("k_cache", c.k_cache), ("ckv_cache", c.ckv_cache), ("k_rope_scale", c.k_scale),
                      ("k_rope_offset", c.k_offset), ("c_kv_scale", c.v_scale), ("c_kv_offset", c.v_offset),
                      ("v_optional", c.v)):
        if arr is not None:
            assert ext[name] == arr.nbytes, name
    rows = c.B * c.N * c.S
    quant = c.k_scale is not None or c.v_scale is not None
    outputs = c.is_output_kv and (c.cache_mode != "Norm" or (c.variant == 2 and quant))
    assert ext["k_rope"] == (rows * c.k_width * 2 if outputs else 0)
    assert ext["c_kv"] == (rows * c.ckv_width * 2 if outputs else 0)
    assert ext["dev_error_count"] == 4


def test_need_refuses_only_short_tensors():
    t = torch.zeros(10, dtype=torch.int16)  # 20 bytes
    native._need(t, 20, "t")
    native._need(t, 8, "t")
    native._need(None, 1 << 40, "absent")
    with pytest.raises(ValueError, match="needs 21 bytes"):
        native._need(t, 21, "t")
    # a byte view counts bytes, not elements of the original dtype
    native._need(t.view(torch.uint8), 20, "t")


def _host(x):
    return runner.to_dev(x, "cpu")


def test_short_kv_cache_is_refused_before_the_device():
    c = synth.make_kv("short", 9, variant=2, B=2, N=2, S=20, Dkv=192, Dv=128, block_size=32, block_num=2,
                      quant_k=True, quant_v=True)
    p = runner.kv_params(c)
    args = dict(kv=_host(c.kv), gamma=_host(c.gamma), cos=_host(c.cos), sin=_host(c.sin),
                index=_host(c.index), k_cache=_host(c.k_cache), ckv_cache=_host(c.ckv_cache),
                k_rope_scale=_host(c.k_scale), c_kv_scale=_host(c.v_scale), k_rope_offset=_host(c.k_offset),
                c_kv_offset=_host(c.v_offset), v_optional=_host(c.v))
    # full-size CPU tensors pass the size checks and stop at the placement check
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        native.kv_rms_norm_rope_cache(p, **args)
    for name in ("kv", "index", "k_cache", "ckv_cache", "c_kv_scale", "v_optional"):
        short = dict(args)
        short[name] = args[name].flatten()[:-1]
        with pytest.raises(ValueError, match=rf"^{name}: the call needs"):
            native.kv_rms_norm_rope_cache(p, **short)


def test_short_qkv_buffers_are_refused_before_the_device():
    c = synth.make_qkv("short", 10, S=16, H=128, num_heads=2, num_kv_heads=2, head_dim=64)
    p = runner.qkv_params(c)
    out = torch.empty((c.T, c.I), dtype=torch.bfloat16)
    packed = torch.empty(native.qkv_cte_mx_packed_weight_bytes(c.H, c.I), dtype=torch.uint8)
    ws = torch.empty(16, dtype=torch.uint8)
    args = [p, _host(c.a), _host(c.a_scale), packed, None, _host(c.bias), _host(c.cos), _host(c.sin),
            _host(c.q_gamma), _host(c.k_gamma), out, ws]
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        native.qkv_cte_mx(*args)
    for pos, name in ((1, "a"), (3, "w_packed"), (6, "cos_cache"), (9, "k_gamma"), (10, "out")):
        short = list(args)
        short[pos] = args[pos].flatten()[:-1]
        with pytest.raises(ValueError, match=rf"^{name}: the call needs"):
            native.qkv_cte_mx(*short)
    with pytest.raises(ValueError, match=r"^out: the call needs"):
        native.qkv_cte_mx_norm_rope(p, _host(c.cos), _host(c.sin), out.flatten()[:-1], ws)
    with pytest.raises(ValueError, match=r"^a_scale: the call needs"):
        native.qkv_cte_mx_project(p, _host(c.a), _host(c.a_scale)[:-1], packed, None, _host(c.bias),
                                  _host(c.q_gamma), _host(c.k_gamma), out, ws)


def test_short_row_quantiser_outputs_are_refused():
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"^codes: the call needs 256 bytes"):
        native.row_quantize_e4m3(x, torch.empty(255, dtype=torch.uint8), torch.empty(4))
    with pytest.raises(ValueError, match=r"^scale: the call needs 16 bytes"):
        native.row_quantize_e4m3(x, torch.empty(256, dtype=torch.uint8), torch.empty(3))
    with pytest.raises(ValueError, match=r"^packed: the call needs 272 bytes"):
        native.row_quantize_e4m3_packed(x, torch.empty(271, dtype=torch.uint8))
