"""The acceptance checker must flag the corruptions the pages describe (no GPU).

ROCm/aiter PR 6539 (Motivation) describes the failure signature: whole 16-64
row bands of an output tile off by one K tile, max relative error ~0.15.
ROCm/mori PR 785 (Test) adds that the corruption can sit near the fp8 floor,
which is why the check is element-wise.  Each corruption below is produced by
the oracle on modified inputs, on the CPU.
"""
import numpy as np
import pytest

import oracle
import synth
from checker import check


def _case(K):
    return synth.make_case("ptpc", 128, 256, K, seed=21, b_std=0.02)


@pytest.mark.parametrize("K", [256, 1792])
def test_clean_output_passes(K):
    c = _case(K)
    _, ref = oracle.gemm("ptpc", *c.numpy())
    assert check(ref, ref)["ok"]


@pytest.mark.parametrize("K,kind", [(256, "drop"), (256, "repeat"), (1792, "drop"), (1792, "repeat")])
def test_band_off_by_one_k_tile_is_flagged(K, kind):
    c = _case(K)
    A, B, sa, sb = c.numpy()
    _, ref = oracle.gemm("ptpc", A, B, sa, sb)
    rows = slice(32, 48)  # a 16-row band
    kt = K // 128 - 1  # the last K tile, the one the races hit
    Am = A.copy()
    if kind == "drop":
        Am[rows, kt * 128:(kt + 1) * 128] = 0
    else:  # the band reads the previous K tile's data again
        Am[rows, kt * 128:(kt + 1) * 128] = A[rows, (kt - 1) * 128:kt * 128]
    _, bad_band = oracle.gemm("ptpc", Am, B, sa, sb, rows=(32, 48))
    out = ref.copy()
    out[rows] = bad_band
    r = check(out, ref)
    assert not r["ok"] and r["bad"] > 0, r


def test_single_nan_is_flagged():
    c = _case(256)
    _, ref = oracle.gemm("ptpc", *c.numpy())
    out = ref.copy()
    out[77, 130] = 0x7FC0
    r = check(out, ref)
    assert not r["ok"] and r["nan"] == 1


def test_single_element_three_percent_off_is_flagged():
    c = _case(256)
    _, ref = oracle.gemm("ptpc", *c.numpy())
    vals = oracle.bits_to_f64(ref)
    i = np.unravel_index(np.argmax(np.abs(vals)), vals.shape)
    out = ref.copy()
    out[i] = oracle.bf16_rne([vals[i] * 1.03])[0]
    r = check(out, ref)
    assert not r["ok"] and r["bad"] == 1


def test_one_ulp_differences_pass():
    c = _case(1792)
    _, ref = oracle.gemm("ptpc", *c.numpy())
    out = ref.copy()
    out[::3, ::5] ^= 1  # flip the last mantissa bit of a third of the elements
    assert check(out, ref)["ok"]
