"""Pins for the oracle's GEMM in every mode (no GPU).

Independent checks: int64 sums of integer-valued operands, exact rational
brute force on tiny shapes (with torch's decoders and an exact nearest-bf16
search), hand-worked examples from tests/golden/, one-hot weights, scale
invariants, transposition, and a float64 library matmul.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from test_oracle_decoders import _nearest_even_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e4m3_codes(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_dec_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_dec_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ---- integer-valued operands: the sum is an integer, computed in int64 --------


@pytest.mark.parametrize("M,N,K,lo,hi", [(17, 23, 256, -16, 16), (5, 7, 4096, -16, 16), (9, 3, 96, -3, 3)])
def test_integer_operands_equal_int64_sum(M, N, K, lo, hi):
    c = synth.make_int_case(M, N, K, lo, hi, seed=M)
    A, B, sa, sb = c.numpy()
    R, ref = oracle.gemm("ptpc", A, B, sa, sb)
    ai = _torch_dec_e4m3(A).astype(np.int64)
    bi = _torch_dec_e4m3(B).astype(np.int64)
    assert np.all(ai == _torch_dec_e4m3(A))  # the operands really are integers
    exact = ai @ bi.T
    assert np.array_equal(R, exact.astype(np.float64))
    lib = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref, lib)


# ---- exact rational brute force on tiny shapes, every mode -------------------


def _brute(case, with_abs=False):
    """Exact rational value of every output (and the sum of |terms| it adds up)."""
    A, B, sa, sb = case.numpy()
    M, N, K = case.M, case.N, case.K
    if case.mode == "bf16":
        a, b = _torch_dec_bf16(A), _torch_dec_bf16(B)
    else:
        a, b = _torch_dec_e4m3(A), _torch_dec_e4m3(B)
    out = [[None] * N for _ in range(M)]
    mag = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            prods = [Fraction(float(a[m, k])) * Fraction(float(b[n, k])) for k in range(K)]
            if case.mode == "bf16":
                terms = prods
            elif case.mode == "ptpc":
                terms = [sum(prods, Fraction(0)) * Fraction(float(sa[m])) * Fraction(float(sb[n]))]
            elif case.mode == "blockscale":
                terms = [
                    sum(prods[128 * j:128 * j + 128], Fraction(0)) * Fraction(float(sa[j, m])) * Fraction(float(sb[n // 128, j]))
                    for j in range(K // 128)
                ]
            else:
                terms = [
                    sum(prods[32 * j:32 * j + 32], Fraction(0))
                    * Fraction(2) ** (int(sa[j, m]) - 127)
                    * Fraction(2) ** (int(sb[j, n]) - 127)
                    for j in range(K // 32)
                ]
            out[m][n] = sum(terms, Fraction(0))
            mag[m][n] = sum((abs(t) for t in terms), Fraction(0))
    return (out, mag) if with_abs else out


@pytest.mark.parametrize(
    "mode,M,N,K",
    [("ptpc", 3, 5, 48), ("ptpc", 4, 2, 256), ("blockscale", 3, 130, 256), ("mxfp8", 4, 5, 128), ("bf16", 3, 4, 40)],
)
def test_tiny_shapes_match_exact_rational_brute_force(mode, M, N, K):
    case = synth.make_case(mode, M, N, K, seed=11, a_std=1.0, b_std=0.5)
    R, ref = oracle.gemm(mode, *case.numpy())
    exact, mag = _brute(case, with_abs=True)
    for m in range(M):
        for n in range(N):
            e = exact[m][n]
            # R is within a few binary64 roundings (relative to the sum of |terms|)
            assert abs(Fraction(float(R[m, n])) - e) <= (mag[m][n] + abs(e)) * Fraction(K + 4, 2**53)
            assert int(ref[m, n]) == _nearest_even_bf16(float(e)), (mode, m, n, float(e), hex(ref[m, n]))


def test_ptpc_and_mxfp8_sums_are_exact():
    # ptpc without scales and mxfp8 (power-of-two scales) are exact in binary64.
    case = synth.make_case("mxfp8", 2, 3, 64, seed=3)
    R, _ = oracle.gemm("mxfp8", *case.numpy())
    exact = _brute(case)
    for m in range(2):
        for n in range(3):
            assert Fraction(float(R[m, n])) == exact[m][n]


# ---- hand-worked examples ------------------------------------------------------


def _parse_matrix(s, rows, cols, as_float=True):
    out = []
    for row in s.split(";"):
        vals = []
        for tok in row.split(","):
            tok = tok.strip()
            if "*" in tok:
                v, n = tok.split("*")
                vals += [float(v) if as_float else int(v)] * int(n)
            else:
                vals.append(float(tok) if as_float else int(tok, 0))
        out.append(vals)
    arr = np.array(out)
    assert arr.shape == (rows, cols), (arr.shape, rows, cols)
    return arr


def _golden_cases():
    for line in open(os.path.join(GOLDEN, "worked_examples.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        yield [f.strip() for f in line.split("|")]


@pytest.mark.parametrize("fields", list(_golden_cases()), ids=lambda f: f[0] + "_" + f[1].replace(" ", "x"))
def test_worked_examples(fields):
    mode, dims, a, b, sa, sb, r, ref = fields
    M, N, K = (int(x) for x in dims.split())
    A = _parse_matrix(a, M, K)
    B = _parse_matrix(b, N, K)
    if mode == "bf16":
        Ac = torch.tensor(A, dtype=torch.float32).bfloat16().view(torch.int16).numpy().view(np.uint16)
        Bc = torch.tensor(B, dtype=torch.float32).bfloat16().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(_torch_dec_bf16(Ac), A)
        sa_a = sb_a = None
    else:
        Ac, Bc = _e4m3_codes(A), _e4m3_codes(B)
        assert np.array_equal(_torch_dec_e4m3(Ac), A)  # the values are exact in e4m3
        if mode == "ptpc":
            sa_a = np.array([float(x) for x in sa.replace(";", ",").split(",")], dtype=np.float32)
            sb_a = np.array([float(x) for x in sb.replace(";", ",").split(",")], dtype=np.float32)
        elif mode == "blockscale":
            sa_a = _parse_matrix(sa, K // 128, M).astype(np.float32)
            sb_a = _parse_matrix(sb, (N + 127) // 128, K // 128).astype(np.float32)
        else:
            sa_a = _parse_matrix(sa, K // 32, M, as_float=False).astype(np.uint8)
            sb_a = _parse_matrix(sb, K // 32, N, as_float=False).astype(np.uint8)
    R, refb = oracle.gemm(mode, Ac, Bc, sa_a, sb_a)
    want_r = _parse_matrix(r, M, N)
    want_ref = _parse_matrix(ref, M, N, as_float=False)
    assert np.array_equal(R, want_r), (R, want_r)
    assert np.array_equal(refb.astype(np.int64), want_ref), ([hex(x) for x in refb.ravel()], want_ref)


# ---- special cases with closed forms ----------------------------------------


def test_one_hot_weights_select_columns():
    # B[n,k] = 1 iff k == perm[n] (K == N): ref[m,n] = bf16(A[m,perm[n]] * sa[m] * sb[n]).
    M = N = K = 64
    rng = np.random.default_rng(5)
    perm = rng.permutation(K)
    case = synth.make_case("ptpc", M, N, K, seed=5)
    A, _, sa, sb = case.numpy()
    B = np.zeros((N, K), dtype=np.uint8)
    B[np.arange(N), perm] = _e4m3_codes([1.0])[0]
    R, ref = oracle.gemm("ptpc", A, B, sa, sb)
    a = _torch_dec_e4m3(A)
    want = a[:, perm] * sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
    assert np.array_equal(R, want)
    # one rounding from binary64 must equal the exact nearest-even search
    for m in range(0, M, 7):
        for n in range(0, N, 5):
            assert int(ref[m, n]) == _nearest_even_bf16(float(want[m, n]))


def test_mxfp8_with_unit_scales_equals_ptpc_with_unit_scales():
    case = synth.make_case("mxfp8", 16, 24, 256, seed=2)
    A, B, _, _ = case.numpy()
    ones_a = np.full((256 // 32, 16), 127, dtype=np.uint8)
    ones_b = np.full((256 // 32, 24), 127, dtype=np.uint8)
    R1, r1 = oracle.gemm("mxfp8", A, B, ones_a, ones_b)
    R2, r2 = oracle.gemm("ptpc", A, B, np.ones(16, np.float32), np.ones(24, np.float32))
    assert np.array_equal(R1, R2) and np.array_equal(r1, r2)


def test_blockscale_with_uniform_power_of_two_scales_equals_ptpc():
    M, N, K = 8, 200, 384
    case = synth.make_case("blockscale", M, N, K, seed=4)
    A, B, _, _ = case.numpy()
    alpha = np.exp2(np.arange(M) % 5 - 2).astype(np.float32)  # per row, same in every K block
    beta = np.float32(0.25)
    sa = np.tile(alpha, (K // 128, 1))
    sb = np.full(((N + 127) // 128, K // 128), beta, dtype=np.float32)
    R1, r1 = oracle.gemm("blockscale", A, B, sa, sb)
    R2, r2 = oracle.gemm("ptpc", A, B, alpha, np.full(N, beta, np.float32))
    assert np.array_equal(R1, R2) and np.array_equal(r1, r2)


def test_doubling_a_scale_doubles_the_result():
    for mode in ("ptpc", "blockscale", "mxfp8"):
        case = synth.make_case(mode, 8, 136, 256, seed=9)
        A, B, sa, sb = case.numpy()
        R1, _ = oracle.gemm(mode, A, B, sa, sb)
        sa2 = (sa + 1).astype(np.uint8) if mode == "mxfp8" else (sa * 2).astype(np.float32)
        R2, _ = oracle.gemm(mode, A, B, sa2, sb)
        assert np.array_equal(R2, 2 * R1), mode


def test_swapping_operands_transposes_ptpc():
    case = synth.make_case("ptpc", 12, 20, 96, seed=6)
    A, B, sa, sb = case.numpy()
    R1, r1 = oracle.gemm("ptpc", A, B, sa, sb)
    R2, r2 = oracle.gemm("ptpc", B, A, sb, sa)
    # (s*sa)*sb vs (s*sb)*sa may differ by one binary64 rounding; bf16 must agree
    assert np.allclose(R1, R2.T, rtol=2**-51, atol=0)
    assert np.array_equal(r1, r2.T)


def test_rows_and_points_agree():
    for mode in ("ptpc", "blockscale", "mxfp8", "bf16"):
        case = synth.make_case(mode, 40, 264, 256, seed=8)
        R, ref = oracle.gemm(mode, *case.numpy())
        R2, ref2 = oracle.gemm(mode, *case.numpy(), rows=(7, 30))
        assert np.array_equal(R[7:30], R2) and np.array_equal(ref[7:30], ref2)
        ms = np.array([0, 39, 13, 7, 22])
        ns = np.array([0, 263, 128, 5, 200])
        Rp, refp = oracle.gemm_points(mode, *case.numpy(), ms, ns)
        assert np.array_equal(Rp, R[ms, ns]) and np.array_equal(refp, ref[ms, ns])


# ---- library cross-check ------------------------------------------------------


@pytest.mark.parametrize("mode", ["ptpc", "blockscale", "mxfp8", "bf16"])
def test_float64_library_matmul(mode):
    M, N, K = 96, 160, 1792 if mode != "bf16" else 512
    case = synth.make_case(mode, M, N, K, seed=12, b_std=0.02)
    A, B, sa, sb = case.numpy()
    R, _ = oracle.gemm(mode, A, B, sa, sb)
    if mode == "bf16":
        want = torch.from_numpy(_torch_dec_bf16(A)) @ torch.from_numpy(_torch_dec_bf16(B)).T
    else:
        a = torch.from_numpy(_torch_dec_e4m3(A))
        b = torch.from_numpy(_torch_dec_e4m3(B))
        if mode == "ptpc":
            a = a * torch.from_numpy(sa.astype(np.float64))[:, None]
            b = b * torch.from_numpy(sb.astype(np.float64))[:, None]
        elif mode == "blockscale":
            a = a * torch.from_numpy(sa.astype(np.float64)).T.repeat_interleave(128, dim=1)
            bs = torch.from_numpy(sb.astype(np.float64)).repeat_interleave(128, dim=0)[:N]
            b = b * bs.repeat_interleave(128, dim=1)
        else:
            a = a * torch.from_numpy(np.exp2(sa.astype(np.float64) - 127)).T.repeat_interleave(32, dim=1)
            b = b * torch.from_numpy(np.exp2(sb.astype(np.float64) - 127)).T.repeat_interleave(32, dim=1)
        want = a @ b.T
    want = want.numpy()
    err = np.abs(R - want).max() / np.abs(want).max()
    assert err <= 1e-12, err


def test_rejects_bad_shapes():
    case = synth.make_case("blockscale", 4, 8, 128, seed=0)
    A, B, sa, sb = case.numpy()
    with pytest.raises(ValueError):
        oracle.gemm("blockscale", A[:, :96], B[:, :96], sa, sb)  # K % 128 != 0
