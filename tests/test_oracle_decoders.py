"""Pins for the oracle's scalar decoders and its bf16 rounding (no GPU).

Each pin is independent of the oracle's own code: torch's float8 / bfloat16
conversions (library routines), the OCP named-value tables under
tests/golden/, and an exact rational nearest-value search.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        rows.append((int(a, 0), float(b)))
    return rows


def _same(x, y):
    if math.isnan(x) or math.isnan(y):
        return math.isnan(x) and math.isnan(y)
    return x == y and math.copysign(1, x) == math.copysign(1, y)


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.dec_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(mine[c], lib[c]), (hex(c), mine[c], lib[c])


def test_e4m3_named_values():
    for code, val in _read_pairs("e4m3fn_named_values.txt"):
        got = float(oracle.dec_e4m3([code])[0])
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val, (hex(code), got, val)


def test_e4m3_finite_values_form_the_expected_grid():
    # 2 NaN codes, 254 finite values; magnitudes are 0..7 * 2^-9 below 2^-6 and
    # 8 values per binade above, the largest 448.
    v = oracle.dec_e4m3(np.arange(256, dtype=np.uint8))
    fin = v[~np.isnan(v)]
    assert fin.size == 254
    pos = np.unique(np.abs(fin))
    assert pos.size == 127  # +0 and -0 share |0|
    assert pos.max() == 448.0
    assert np.all(np.diff(pos) > 0)


def test_e8m0_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.dec_e8m0(codes)
    if hasattr(torch, "float8_e8m0fnu"):
        lib = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
        for c in range(256):
            assert _same(mine[c], lib[c]), (c, mine[c], lib[c])
    for c in range(255):
        assert mine[c] == 2.0 ** (c - 127)
    assert math.isnan(mine[255])


def test_e8m0_named_values():
    for code, val in _read_pairs("e8m0_named_values.txt"):
        got = float(oracle.dec_e8m0([code])[0])
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val, (code, got, val)


def test_bf16_decoder_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    mine = oracle.dec_bf16(bits)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for a, b in zip(mine, lib):
        assert _same(a, b)


def test_bf16_rne_on_float32_values_matches_torch():
    # For inputs that are exactly float32 values, one rounding from binary64
    # equals torch's float32 -> bfloat16 (round-to-nearest-even).
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # add every tie pattern in a few binades and around the subnormal range
    ties = np.array([(e << 23) | (m << 16) | 0x8000 for e in (1, 2, 100, 127, 128, 200, 254) for m in range(0, 128, 3)], dtype=np.uint32)
    subs = np.arange(0, 1 << 17, 97, dtype=np.uint32)
    bits = np.concatenate([bits, ties, ties | 0x80000000, subs])
    f32 = bits.view(np.float32)
    fin = np.isfinite(f32)
    f32 = f32[fin]
    mine = oracle.bf16_rne(f32.astype(np.float64))
    lib = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(mine != lib)[0]
    assert bad.size == 0, [(float(f32[i]), hex(mine[i]), hex(lib[i])) for i in bad[:5]]


def test_bf16_rne_hand_ties():
    assert oracle.bf16_rne([1 + 2**-8])[0] == 0x3F80  # tie -> even (1.0)
    assert oracle.bf16_rne([1 + 3 * 2**-8])[0] == 0x3F82  # tie -> even (1 + 2^-6)
    assert oracle.bf16_rne([1 + 2**-8 + 2**-40])[0] == 0x3F81  # just above the tie
    assert oracle.bf16_rne([-(1 + 2**-8)])[0] == 0xBF80
    assert oracle.bf16_rne([0.0])[0] == 0x0000
    assert oracle.bf16_rne([-0.0])[0] == 0x8000
    assert oracle.bf16_rne([2.0**-133])[0] == 0x0001  # smallest bf16 subnormal
    assert oracle.bf16_rne([2.0**-134])[0] == 0x0000  # tie at half of it -> even (0)
    assert oracle.bf16_rne([3 * 2.0**-135])[0] == 0x0001
    assert oracle.bf16_rne([2.0**200])[0] == 0x7F80
    assert oracle.bf16_rne([float("nan")])[0] == 0x7FC0


_BF16_TABLE = None


def _bf16_sorted():
    """All finite bf16 values (decoded by torch) sorted, with their codes."""
    global _BF16_TABLE
    if _BF16_TABLE is None:
        codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        vals = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        keep = np.isfinite(vals) & ~((vals == 0) & (codes == 0x8000))
        vals, codes = vals[keep], codes[keep]
        order = np.argsort(vals, kind="stable")
        _BF16_TABLE = (vals[order], codes[order])
    return _BF16_TABLE


def _nearest_even_bf16(x: float) -> int:
    """Exact rational search: the finite bf16 value nearest to x, ties to even code."""
    vals, codes = _bf16_sorted()
    i = int(np.searchsorted(vals, x))
    cands = [j for j in (i - 1, i) if 0 <= j < vals.size]
    fx = Fraction(x)
    best = min(abs(Fraction(float(vals[j])) - fx) for j in cands)
    win = [j for j in cands if abs(Fraction(float(vals[j])) - fx) == best]
    if len(win) == 2:
        win = [j for j in win if (int(codes[j]) & 1) == 0]
    code = int(codes[win[0]])
    if x < 0 and code == 0:
        code = 0x8000
    return code


def test_bf16_rne_on_binary64_values_matches_exact_search():
    # Values that are not float32 values: a path through float32 would round twice.
    rng = np.random.default_rng(7)
    xs = list(rng.standard_normal(3000) * np.exp2(rng.integers(-30, 30, size=3000)))
    # values a hair above/below bf16 ties, where double rounding would differ
    for m in range(0, 128, 5):
        t = (1 + (2 * m + 1) * 2.0**-8)
        xs += [t + 2.0**-40, t - 2.0**-40, -(t + 2.0**-30)]
    xs = np.array(xs, dtype=np.float64)
    mine = oracle.bf16_rne(xs)
    for x, got in zip(xs, mine):
        assert int(got) == _nearest_even_bf16(float(x)), (x, hex(got))
