"""Teeth for the oracle's pins: plant a plausible mistake in a copy of oracle.c
(on the CPU), build it, and require that at least one pin fails against it.

The mutants cover a wrong exponent bias, a wrong subnormal scale, a lost sign,
a dropped scale, a dropped term, wrong block / scale indices and ties rounded
away from even.  The copy lives in a temporary directory; the real oracle is
untouched.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_decoders as dec
import test_oracle_gemm as gem
import test_oracle_quantize as qnt

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "exponent_bias": ("v = ldexp(1.0 + (double)f / 8.0, e - 7);", "v = ldexp(1.0 + (double)f / 8.0, e - 8);"),
    "subnormal_scale": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "lost_sign": ("return s ? -v : v;", "return v;"),
    "dropped_row_scale": ("return s * (double)((const float*)sa)[m] * (double)((const float*)sb)[n];", "return s * (double)((const float*)sb)[n];"),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];", "for (int64_t k = 0; k + 1 < K; ++k) s += a[k] * b[k];"),
    "block_short_by_one": ("for (int64_t k = j * bk; k < (j + 1) * bk; ++k)", "for (int64_t k = j * bk; k + 1 < (j + 1) * bk; ++k)"),
    "weight_block_index": ("s_b = (double)((const float*)sb)[(n / 128) * nblk + j];", "s_b = (double)((const float*)sb)[j];"),
    "act_block_index": ("s_a = (double)((const float*)sa)[j * M + m];", "s_a = (double)((const float*)sa)[m];"),
    "mx_scale_index": ("s_b = sgo_dec_e8m0(((const uint8_t*)sb)[j * N + n]);", "s_b = sgo_dec_e8m0(((const uint8_t*)sb)[n]);"),
    "ties_away": ("if (rem > half || (rem == half && (n & 1))) n += 1;", "if (rem >= half) n += 1;"),
    "bf16_decode_shift": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;"),
    "e4m3_ties_away": ("if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;", "if (rem >= 0.5) fl += 1.0;"),
    "mx_exponent_off_by_one": ("    while (448.0 * ldexp(1.0, e - 1) >= amax) --e;\n    return e;", "    while (448.0 * ldexp(1.0, e - 1) >= amax) --e;\n    return e + 1;"),
    "quant_scale_448": ("volatile float num = amax, den = 448.0f;", "volatile float num = amax, den = 480.0f;"),
}


def _pins():
    """The pins, as zero-argument callables."""
    yield dec.test_e4m3_all_codes_match_torch
    yield dec.test_e8m0_all_codes
    yield dec.test_bf16_decoder_matches_torch
    yield dec.test_bf16_rne_hand_ties
    yield lambda: gem.test_integer_operands_equal_int64_sum(17, 23, 256, -16, 16)
    for args in [("ptpc", 3, 5, 48), ("blockscale", 3, 130, 256), ("mxfp8", 4, 5, 128), ("bf16", 3, 4, 40)]:
        yield (lambda a=args: gem.test_tiny_shapes_match_exact_rational_brute_force(*a))
    for fields in gem._golden_cases():
        yield (lambda f=fields: gem.test_worked_examples(f))
    for mode in ("ptpc", "blockscale", "mxfp8", "bf16"):
        yield (lambda m=mode: gem.test_float64_library_matmul(m))
    yield qnt.test_e4m3_rounding_matches_torch_within_range
    yield qnt.test_e4m3_ties_and_saturation
    yield qnt.test_ptpc_quantisation_equals_the_input_generator_on_float32
    yield qnt.test_mx_exponent_is_the_least_power_that_covers_amax


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site vanished: " + name
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "libm.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
        real = oracle.lib()
        mut = ctypes.CDLL(so)
        for fn in ("sgo_dec_e4m3", "sgo_dec_e8m0", "sgo_dec_bf16", "sgo_bf16_rne", "sgo_gemm_rows", "sgo_gemm_points", "sgo_num_threads", "sgo_e4m3_rne_sat", "sgo_quantize"):
            getattr(mut, fn).restype = getattr(real, fn).restype
            getattr(mut, fn).argtypes = getattr(real, fn).argtypes
        monkeypatch.setattr(oracle, "_lib", mut)
        caught = 0
        for pin in _pins():
            try:
                pin()
            except (AssertionError, ValueError):
                caught += 1
                break
        assert caught, "no pin failed for mutant " + name
