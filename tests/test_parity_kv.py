"""GPU parity: kv_rms_norm_rope_cache (C-ABI) against the fp64 oracle.

Small cases span several warps, ragged row counts, both variants, both paged
layouts, bf16 and int8 caches, symmetric and asymmetric quantisation, skipped
(-1) and out-of-range slots.  The full-size DeepSeek-V3 MLA (V1) and separate
k/v (V2) workloads are compared element by element over every output.
"""
import numpy as np
import pytest
import torch

from parity_util import check_kv
from rope_attention_gb300 import runner, synth

pytestmark = pytest.mark.gpu


def run_case(case):
    r = runner.KvRun(case)
    r.run()
    torch.cuda.synchronize()
    return r


SMALL = [
    # name, kwargs
    ("v1_bf16_bnsd", dict(variant=1, B=3, N=1, S=37, Dkv=576, Dv=512, block_size=16, block_num=8)),
    ("v1_int8_bnsd", dict(variant=1, B=2, N=1, S=45, Dkv=576, Dv=512, block_size=32, block_num=4,
                          quant_k=True, quant_v=True)),
    ("v1_int8_sym", dict(variant=1, B=2, N=1, S=33, Dkv=576, Dv=512, block_size=32, block_num=4,
                         quant_k=True, quant_v=True, offsets=False)),
    ("v1_kq_only", dict(variant=1, B=2, N=1, S=20, Dkv=576, Dv=512, block_size=32, block_num=2,
                        quant_k=True)),
    ("v1_pa", dict(variant=1, B=2, N=1, S=19, Dkv=576, Dv=512, block_size=16, block_num=4,
                   cache_mode="PA")),
    ("v1_small_dims", dict(variant=1, B=2, N=1, S=11, Dkv=136, Dv=128, rope_size=8, block_size=16,
                           block_num=2)),
    ("v2_int8_bnsd", dict(variant=2, B=2, N=8, S=29, Dkv=192, Dv=128, block_size=32, block_num=4,
                          quant_k=True, quant_v=True)),
    ("v2_bf16_pa", dict(variant=2, B=3, N=4, S=21, Dkv=192, Dv=128, block_size=16, block_num=8,
                        cache_mode="PA")),
    ("v2_vq_only_n2", dict(variant=2, B=2, N=2, S=40, Dkv=192, Dv=128, block_size=32, block_num=4,
                           quant_v=True)),
    ("v2_n1_wide", dict(variant=2, B=1, N=1, S=50, Dkv=384, Dv=256, block_size=16, block_num=4)),
    # several rows per warp step: groups that cross head and batch boundaries (S smaller
    # than the rows a warp handles at once), and fewer rows than lanes
    ("v2_s1_n8", dict(variant=2, B=3, N=8, S=1, Dkv=192, Dv=128, block_size=32, block_num=1,
                      quant_k=True, quant_v=True)),
    ("v2_s3_n8_narrow", dict(variant=2, B=2, N=8, S=3, Dkv=64, Dv=64, block_size=32, block_num=1,
                             quant_k=True)),
    # block_size that is not a power of two (division path for the slot)
    ("v2_bs48", dict(variant=2, B=2, N=2, S=30, Dkv=192, Dv=128, block_size=48, block_num=3)),
    # every lane of the row holds RoPE pairs
    ("v2_rope256", dict(variant=2, B=1, N=2, S=20, Dkv=256, Dv=64, rope_size=256, block_size=32,
                        block_num=1, quant_k=True, quant_v=True)),
    # v wider than kv, small rope
    ("v2_v_wider", dict(variant=2, B=2, N=1, S=13, Dkv=64, Dv=512, rope_size=32, block_size=32,
                        block_num=1, quant_v=True)),
    # rms_size 1024: four chunks per lane at 32 lanes per row
    ("v1_wide", dict(variant=1, B=1, N=1, S=17, Dkv=1088, Dv=1024, block_size=32, block_num=1,
                     quant_k=True, quant_v=True)),
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("skip", [0.0, 0.25])
def test_small(name, kw, skip):
    case = synth.make_kv(name, 100 + len(name), skip_frac=skip, **kw)
    check_kv(case, run_case(case), name)


VARIANTS = [
    # Norm cache mode: [B, N, Scache, D], index [B, S] of per-batch offsets
    ("norm_v2_int8", dict(variant=2, B=3, N=4, S=37, Dkv=192, Dv=128, cache_mode="Norm", cache_seq=50,
                          quant_k=True, quant_v=True)),
    ("norm_v2_bf16_no_outputs", dict(variant=2, B=2, N=2, S=20, Dkv=192, Dv=128, cache_mode="Norm",
                                     cache_seq=24)),
    ("norm_v1_bf16", dict(variant=1, B=3, N=1, S=21, Dkv=576, Dv=512, cache_mode="Norm", cache_seq=21)),
    # PA_BLK_BNSD: one start slot per block of block_size tokens; partial last block
    ("blk_v2_int8", dict(variant=2, B=2, N=2, S=70, Dkv=192, Dv=128, block_size=32,
                         cache_mode="PA_BLK_BNSD", quant_k=True, quant_v=True)),
    ("blk_v1_bf16_bs48", dict(variant=1, B=2, N=1, S=100, Dkv=576, Dv=512, block_size=48,
                              cache_mode="PA_BLK_BNSD")),
    # cos/sin [B, N, 1, R] broadcast over S
    ("bcast_v2_int8", dict(variant=2, B=2, N=8, S=29, Dkv=192, Dv=128, block_size=32, block_num=4,
                           quant_k=True, quant_v=True, rope_broadcast=True)),
    ("bcast_norm_v1", dict(variant=1, B=2, N=1, S=33, Dkv=576, Dv=512, cache_mode="Norm",
                           cache_seq=40, rope_broadcast=True)),
    # fp16 inputs (and fp16 caches / outputs when not quantised)
    ("fp16_v1", dict(variant=1, B=2, N=1, S=45, Dkv=576, Dv=512, block_size=16, block_num=8, dtype="fp16")),
    ("fp16_v2_int8_k", dict(variant=2, B=2, N=4, S=30, Dkv=192, Dv=128, block_size=32, block_num=2,
                            dtype="fp16", quant_k=True)),
    ("fp16_v2_pa", dict(variant=2, B=3, N=2, S=21, Dkv=192, Dv=128, block_size=16, block_num=4,
                        dtype="fp16", cache_mode="PA")),
    # FP8 caches
    ("fp8_v2_e4m3_e5m2", dict(variant=2, B=2, N=8, S=29, Dkv=192, Dv=128, block_size=32, block_num=4,
                              quant_k=True, quant_v=True, k_qtype="e4m3", v_qtype="e5m2")),
    ("fp8_v1_e5m2_sym", dict(variant=1, B=2, N=1, S=45, Dkv=576, Dv=512, block_size=32, block_num=4,
                             quant_k=True, quant_v=True, k_qtype="e5m2", v_qtype="e4m3", offsets=False)),
    ("fp8_fp16_norm_v2", dict(variant=2, B=2, N=2, S=40, Dkv=192, Dv=128, cache_mode="Norm", cache_seq=40,
                              dtype="fp16", quant_k=True, quant_v=True, k_qtype="e4m3", v_qtype="int8")),
    # V1 quantisation parameters of shape [1]: pipelined (576/64 int8), register (other dims), FP8
    ("scalar_v1_int8", dict(variant=1, B=2, N=1, S=45, Dkv=576, Dv=512, block_size=32, block_num=4,
                            quant_k=True, quant_v=True, k_scalar=True, v_scalar=True)),
    ("scalar_v1_k_only_sym", dict(variant=1, B=2, N=1, S=33, Dkv=576, Dv=512, block_size=32, block_num=4,
                                  quant_k=True, quant_v=True, k_scalar=True, offsets=False)),
    ("scalar_v1_small_dims", dict(variant=1, B=2, N=1, S=21, Dkv=136, Dv=128, rope_size=8, block_size=32,
                                  block_num=2, quant_k=True, quant_v=True, k_scalar=True, v_scalar=True)),
    ("scalar_fp8_v1", dict(variant=1, B=2, N=1, S=30, Dkv=576, Dv=512, block_size=32, block_num=2,
                           quant_k=True, quant_v=True, k_qtype="e4m3", v_qtype="e5m2", v_scalar=True)),
]


@pytest.mark.parametrize("name,kw", VARIANTS, ids=[s[0] for s in VARIANTS])
@pytest.mark.parametrize("skip", [0.0, 0.2])
def test_variants(name, kw, skip):
    case = synth.make_kv(name, 400 + len(name), skip_frac=skip, **kw)
    if "fp8" in name and case.k_scale is not None:
        case.k_scale *= 8.0  # drive some codes into saturation
    check_kv(case, run_case(case), name)


def test_norm_mode_repeated_offsets_and_bad_values():
    """Norm mode: the same offsets in different batches are legal; an offset outside
    [-1, Scache) is counted once per token and not written."""
    case = synth.make_kv("norm_bad", 9, variant=2, B=3, N=2, S=16, Dkv=192, Dv=128, cache_mode="Norm",
                         cache_seq=20, quant_k=True, quant_v=True)
    case.index[1] = case.index[0]
    case.index[2, 3] = 20
    case.index[0, 5] = -3
    check_kv(case, run_case(case), "norm-bad")


def test_blk_mode_skipped_and_bad_blocks():
    case = synth.make_kv("blk_bad", 10, variant=2, B=2, N=2, S=50, Dkv=192, Dv=128, block_size=16,
                         cache_mode="PA_BLK_BNSD")
    case.index[1] = -1                                       # a whole block skipped
    case.index[4] = case.block_num * case.block_size - 3     # block runs past the end of the cache
    check_kv(case, run_case(case), "blk-bad")


def test_out_of_range_index_counted_not_written():
    case = synth.make_kv("bad", 7, variant=2, B=2, N=2, S=16, Dkv=192, Dv=128, block_size=16,
                         block_num=4, skip_frac=0.1)
    case.index[3] = case.block_num * case.block_size + 5
    case.index[9] = -4
    check_kv(case, run_case(case), "bad-index")


def test_no_output_kv():
    case = synth.make_kv("nokv", 8, variant=1, B=2, N=1, S=24, Dkv=576, Dv=512, block_size=16,
                         block_num=4, is_output_kv=False)
    check_kv(case, run_case(case), "no-output-kv")


@pytest.mark.parametrize("quant", [False, True], ids=["bf16", "int8"])
def test_full_mla_v1(quant):
    """kv [32,1,4096,576], PA_BNSD bs=128, 131072 slots, is_output_kv."""
    case = synth.kv_mla_v1(quant=quant)
    stats = check_kv(case, run_case(case), "mla_v1")
    print("tie differences:", stats)


def test_full_sep_v2():
    """kv [8,8,4096,192], v [8,8,4096,128], int8 per-head quantisation, PA_BNSD bs=128."""
    case = synth.kv_sep_v2(is_output_kv=True)
    stats = check_kv(case, run_case(case), "sep_v2")
    print("tie differences:", stats)


def test_repeat_call_is_idempotent():
    case = synth.make_kv("rep", 9, variant=1, B=2, N=1, S=64, Dkv=576, Dv=512, block_size=32,
                         block_num=4, quant_k=True, quant_v=True)
    r = run_case(case)
    first = r.k_cache.clone(), r.ckv_cache.clone()
    r.run()
    torch.cuda.synchronize()
    assert torch.equal(first[0], r.k_cache) and torch.equal(first[1], r.ckv_cache)


# The configuration the bench times for the KV half of the 720p step: V2 separate
# k/v, PA_BNSD, int8 per-head quantisation, is_output_kv off (the CANN parameter
# table's default), so the kernel takes its no-outputs branch.
OUTPUTS_OFF = [
    ("v2_int8_off", dict(variant=2, B=2, N=8, S=29, Dkv=192, Dv=128, block_size=32, block_num=4,
                         quant_k=True, quant_v=True)),
    # rows per warp step crossing head and batch boundaries; fewer rows than a tile
    ("v2_int8_off_s3", dict(variant=2, B=3, N=8, S=3, Dkv=192, Dv=128, block_size=32, block_num=1,
                            quant_k=True, quant_v=True)),
    # a ragged tail of rows after several full 16-row tiles of the pipelined kernel
    ("v2_int8_off_ragged", dict(variant=2, B=2, N=4, S=203, Dkv=192, Dv=128, block_size=128,
                                block_num=4, quant_k=True, quant_v=True)),
    ("v2_int8_off_sym_n1", dict(variant=2, B=3, N=1, S=77, Dkv=192, Dv=128, block_size=64,
                                block_num=4, quant_k=True, quant_v=True, offsets=False)),
]


@pytest.mark.parametrize("name,kw", OUTPUTS_OFF, ids=[s[0] for s in OUTPUTS_OFF])
@pytest.mark.parametrize("skip", [0.0, 0.25])
def test_v2_outputs_off(name, kw, skip):
    case = synth.make_kv(name, 600 + len(name), skip_frac=skip, is_output_kv=False, **kw)
    run = runner.KvRun(case)
    assert not run.outputs
    # k_rope / c_kv buffers handed over although is_output_kv is off: the call must
    # leave them alone (the page writes them only when is_output_kv is set)
    fdt = torch.bfloat16
    sentinel = torch.tensor(synth.K_SENTINEL_BF16, dtype=torch.int16)
    run.k_rope = torch.full((case.B, case.N, case.S, case.k_width), 0, dtype=fdt, device="cuda")
    run.c_kv = torch.full((case.B, case.N, case.S, case.ckv_width), 0, dtype=fdt, device="cuda")
    run.k_rope.view(torch.int16).fill_(sentinel.item())
    run.c_kv.view(torch.int16).fill_(sentinel.item())
    run.run()
    torch.cuda.synchronize()
    for t in (run.k_rope, run.c_kv):
        assert bool((t.view(torch.int16) == sentinel.item()).all()), f"{name}: an output was written"
    run.k_rope = run.c_kv = None  # check_kv compares the outputs only when they are on
    check_kv(case, run, name)


def test_full_sep_v2_outputs_off():
    """The benched call itself: kv [8,8,4096,192], v [8,8,4096,128], int8 per-head
    quantisation, PA_BNSD bs=128, 256 blocks, is_output_kv off; every cache slot
    compared (written slots against the oracle, the rest bit for bit)."""
    case = synth.kv_sep_v2(is_output_kv=False)
    stats = check_kv(case, run_case(case), "sep_v2_outputs_off")
    print("tie differences:", stats)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_every_slot_skipped():
    """index all -1: no cache slot is written (every one keeps its sentinel), while the
    k_rope / c_kv outputs are still written for every row."""
    case = synth.make_kv("all_skip", 12, variant=2, B=2, N=4, S=50, Dkv=192, Dv=128, block_size=32,
                         block_num=4, quant_k=True, quant_v=True, skip_frac=1.0)
    assert (case.index == -1).all()
    run = run_case(case)
    assert run.outputs
    check_kv(case, run, "all-skipped")


@pytest.mark.parametrize("variant", [1, 2])
def test_zero_huge_and_tiny_rows(variant):
    """Rows of zeros (RMS 0, so eps alone), rows scaled by 1e15 (int8 codes saturate at
    -128 / 127) and by 1e-15 (eps dominates the RMS), through the pipelined kernel."""
    kw = (dict(variant=1, B=2, N=1, S=40, Dkv=576, Dv=512) if variant == 1
          else dict(variant=2, B=2, N=8, S=40, Dkv=192, Dv=128))
    case = synth.make_kv(f"extreme_v{variant}", 13, block_size=32, block_num=(3 if variant == 1 else 20),
                         quant_k=True, quant_v=True, **kw)
    kv = _bf16_values(case.kv)
    kv[:, :, 0:5] = 0
    kv[:, :, 5:10] *= np.float32(1e15)
    kv[:, :, 10:15] *= np.float32(1e-15)
    case.kv[:] = synth.encode_bf16(kv)
    if case.v is not None:
        v = _bf16_values(case.v)
        v[:, :, 5:10] *= np.float32(1e15)
        case.v[:] = synth.encode_bf16(v)
    check_kv(case, run_case(case), f"extreme-v{variant}")
