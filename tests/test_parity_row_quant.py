"""GPU parity: the row FP8 quantiser (C-ABI) against the oracle, bit for bit.

The codes are integers decided by fp32 arithmetic, and the scales are fp32 values
of the same definition, so both must match the oracle exactly.  Cases span one
to many warps per launch, rows that fill part of a warp, the register path and
the two-pass path for long rows (H > 8192), rows of zeros and of bf16
subnormals, huge and tiny magnitudes, and the packed [T, H + 4] layout.  The
full-size 720p hidden state [75600, 5120] is checked on sampled rows plus
properties every row must have.
"""
import numpy as np
import pytest
import torch

import oracle
from rope_attention_gb300 import native, runner, synth

pytestmark = pytest.mark.gpu


def run_split(bits):
    x = runner.to_dev(bits)
    T, H = bits.shape
    codes = torch.full((T, H), 0x55, dtype=torch.uint8, device="cuda")
    scale = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    native.row_quantize_e4m3(x, codes, scale)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scale.cpu().numpy()


def run_packed(bits):
    x = runner.to_dev(bits)
    T, H = bits.shape
    packed = torch.full((T, H + 4), 0x55, dtype=torch.uint8, device="cuda")
    native.row_quantize_e4m3_packed(x, packed)
    torch.cuda.synchronize()
    return packed.cpu().numpy()


def special_rows(H):
    rng = np.random.default_rng(40)
    rows = [np.zeros(H, np.uint16)]                                   # zeros
    r = np.zeros(H, np.uint16); r[::7] = 0x8000; rows.append(r)       # zeros and negative zeros
    r = np.zeros(H, np.uint16); r[:5] = [0x0001, 0x8002, 0x007F, 0x0040, 0x8001]; rows.append(r)  # subnormals
    rows.append(synth.encode_bf16((rng.normal(0, 1, H) * 1e30).astype(np.float32)))   # huge
    rows.append(synth.encode_bf16((rng.normal(0, 1, H) * 1e-30).astype(np.float32)))  # tiny
    r = synth.encode_bf16(rng.normal(0, 1, H).astype(np.float32)); r[3] = synth.encode_bf16(np.float32([3e38]))[0]
    rows.append(r)                                                    # one dominant element
    return np.stack(rows)


CASES = [("t1_h8", 1, 8), ("t37_h256", 37, 256), ("t300_h5120", 300, 5120), ("t9_h16", 9, 16),
         ("t17_h8192", 17, 8192), ("t6_h8200_twopass", 6, 8200), ("t3_h20480_twopass", 3, 20480),
         ("t65_h1032", 65, 1032)]


@pytest.mark.parametrize("name,T,H", CASES, ids=[c[0] for c in CASES])
def test_split_and_packed_match_oracle(name, T, H):
    bits = synth.hidden_bf16(50 + T, T, H)
    if H >= 16:
        bits = np.concatenate([bits, special_rows(H)])
    codes, scale = run_split(bits)
    c_ref, s_ref = oracle.row_quantize(bits)
    assert np.array_equal(codes, c_ref), f"{name}: {np.count_nonzero(codes != c_ref)} codes differ"
    assert np.array_equal(scale.view(np.uint32), s_ref.view(np.uint32)), f"{name}: scales differ"
    packed = run_packed(bits)
    assert np.array_equal(packed, oracle.row_quantize_packed(bits)), f"{name}: packed rows differ"


def test_full_size_720p_hidden_state():
    """[75600, 5120]: 1024 sampled rows bit for bit; every row has a code of magnitude
    448 at its largest element, and scale = the oracle's scale of that row's amax."""
    T, H = 75600, 5120
    bits = synth.hidden_bf16(4, T, H)
    codes, scale = run_split(bits)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(T - 8, T),
                                     np.random.default_rng(41).choice(T, 1008, replace=False)]))
    c_ref, s_ref = oracle.row_quantize(bits[rows])
    assert np.array_equal(codes[rows], c_ref)
    assert np.array_equal(scale[rows], s_ref)
    absb = bits & np.uint16(0x7FFF)
    top = np.argmax(absb, axis=1)
    assert np.all((codes[np.arange(T), top] & 0x7F) == 0x7E)
    assert not np.any((codes & 0x7F) == 0x7F)  # no NaN codes


def test_every_row_maximum_and_the_magnitudes_below_it():
    """The quotient |x| / scale decides each code.  Every row maximum m the quantiser
    can meet (each positive finite bf16 value >= 2^-100, the amax floor) gets a row
    holding m and every bf16 magnitude in the 20 binades below it -- all the values
    whose code can be nonzero (|x| / scale >= 2^-10 needs |x| >= m * 2^-18.8) -- and
    256 smaller ones, with random signs: 29184 rows x 2816 values, codes and scales
    bit for bit against the oracle."""
    m_bits = np.arange(27 << 7, 0x7F80, dtype=np.int64)          # 2^-100 .. largest finite
    below = np.arange(2816, dtype=np.int64)
    mag = np.maximum(m_bits[:, None] - below[None, :], 0)
    sign = np.random.default_rng(42).integers(0, 2, mag.shape, dtype=np.int64) << 15
    bits = (mag | sign).astype(np.uint16)
    codes, scale = run_split(bits)
    c_ref, s_ref = oracle.row_quantize(bits)
    bad = codes != c_ref
    assert not bad.any(), f"{int(bad.sum())} codes differ; first at {np.argwhere(bad)[0]}"
    assert np.array_equal(scale.view(np.uint32), s_ref.view(np.uint32))
