"""Pins for the oracle's quantisation step (no GPU).

The e4m3 rounding is pinned to torch's float -> float8_e4m3fn conversion (a
library routine; round to nearest even) on every value it can represent and to
hand-checked saturation and tie cases; the scale rules to their definitions by
exact rational checks; the whole per-row quantisation of float32 input to the
seeded input generator's quantiser (which uses torch division and conversion).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rounding_matches_torch_within_range():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000)),
        np.linspace(-447.9, 447.9, 4001),
    ]).astype(np.float32)
    v = v[np.abs(v) < 464]  # torch does not saturate; beyond the top tie it differs by design
    mine = oracle.e4m3_rne_sat(v.astype(np.float64))
    lib = _torch_e4m3(v)
    lib = np.where(np.abs(v) >= 448, np.where(v < 0, 0xFE, 0x7E), lib).astype(np.uint8)
    bad = np.nonzero(mine != lib)[0]
    assert bad.size == 0, [(float(v[i]), hex(mine[i]), hex(lib[i])) for i in bad[:5]]


def test_e4m3_every_code_value_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.dec_e4m3(codes)
    back = oracle.e4m3_rne_sat(vals)
    # +0 and -0 both come back as themselves
    assert np.array_equal(back, codes)


def test_e4m3_ties_and_saturation():
    # ties between neighbouring codes go to the even mantissa
    assert oracle.e4m3_rne_sat([1.0625])[0] == 0x38      # 1 and 1.125: even is 1.0
    assert oracle.e4m3_rne_sat([1.1875])[0] == 0x3A      # 1.125 and 1.25: even is 1.25
    assert oracle.e4m3_rne_sat([2.0 ** -10])[0] == 0x00  # half of the smallest subnormal -> 0
    assert oracle.e4m3_rne_sat([3 * 2.0 ** -10])[0] == 0x02
    assert oracle.e4m3_rne_sat([448.0])[0] == 0x7E
    assert oracle.e4m3_rne_sat([460.0])[0] == 0x7E
    assert oracle.e4m3_rne_sat([1e30])[0] == 0x7E
    assert oracle.e4m3_rne_sat([-1e30])[0] == 0xFE
    assert oracle.e4m3_rne_sat([-0.0])[0] == 0x80


def test_ptpc_quantisation_equals_the_input_generator_on_float32():
    g = torch.Generator("cpu")
    g.manual_seed(9)
    x = torch.randn(64, 512, generator=g) * 3
    x[5] = 0  # an all-zero row takes scale 1
    q_lib, s_lib = synth.quantize_e4m3_rows(x)
    q, s = oracle.quantize("ptpc", x.numpy())
    assert np.array_equal(s, s_lib.numpy())
    assert np.array_equal(q, q_lib.numpy())


def test_blockscale_quantisation_equals_the_input_generator_on_float32():
    g = torch.Generator("cpu")
    g.manual_seed(10)
    x = torch.randn(48, 384, generator=g)
    q_lib, s_lib = synth.quantize_e4m3_blocks_1x128(x)
    q, s = oracle.quantize("blockscale", x.numpy())
    assert np.array_equal(s, s_lib.numpy())
    assert np.array_equal(q, q_lib.numpy())


def test_mx_exponent_is_the_least_power_that_covers_amax():
    g = torch.Generator("cpu")
    g.manual_seed(11)
    x = (torch.randn(40, 256, generator=g) * torch.exp2(torch.randint(-20, 20, (40, 1), generator=g).float())).numpy()
    x[3, :32] = 448.0 * 4  # amax exactly 448 * 2^2
    x[4, :32] = 0.0        # all-zero block
    q, s = oracle.quantize("mxfp8", x)
    for r in range(40):
        for j in range(256 // 32):
            amax = Fraction(float(np.abs(x[r, 32 * j:32 * j + 32]).max()))
            e = int(s[j, r]) - 127
            if amax == 0:
                assert e == 0
                continue
            assert amax <= 448 * Fraction(2) ** e, (r, j)
            assert amax > 448 * Fraction(2) ** (e - 1), (r, j)
    assert int(s[0, 3]) - 127 == 2


def test_quantised_values_reconstruct_within_half_a_code():
    # |x - s * dec(q)| <= s * (half the e4m3 quantum at |x / s|), for every mode
    g = torch.Generator("cpu")
    g.manual_seed(12)
    x = torch.randn(16, 256, generator=g).numpy() * 5
    for mode in ("ptpc", "blockscale", "mxfp8"):
        q, s = oracle.quantize(mode, x)
        d = oracle.dec_e4m3(q)
        if mode == "ptpc":
            sc = s.astype(np.float64)[:, None]
        elif mode == "blockscale":
            sc = np.repeat(s.T.astype(np.float64), 128, axis=1)
        else:
            sc = np.repeat(np.exp2(s.T.astype(np.float64) - 127), 32, axis=1)
        y = x.astype(np.float64) / sc
        quantum = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -9))), -6) - 3)
        assert np.all(np.abs(y - d) <= quantum / 2 + 1e-12 * np.abs(y)), mode
        assert np.all(np.abs(d) <= 448)


def test_bf16_input_equals_float32_input_of_the_same_values():
    g = torch.Generator("cpu")
    g.manual_seed(13)
    xb = torch.randn(8, 128, generator=g).bfloat16()
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    for mode in ("ptpc", "blockscale", "mxfp8"):
        q1, s1 = oracle.quantize(mode, bits)
        q2, s2 = oracle.quantize(mode, xb.float().numpy())
        assert np.array_equal(q1, q2) and np.array_equal(s1, s2), mode
