"""GPU parity for the quantisation step (scaled_gemm_quantize through the C ABI)
against the CPU oracle.  Codes and scales are integers decided by the same fp32
operations on both sides (IEEE division, round to nearest even with
saturation, an exact power-of-two rule for e8m0), so they must match bit for
bit.  Cited: ROCm/mori PR 809, "Using it" (quantize_per_token before the GEMM)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util

    gpu_util.lib_ready()
    from fp8_scaled_gemm_sm_gb300 import binding

    return binding


def _make(R, C, seed, dtype):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    x = torch.randn(R, C, generator=g) * torch.exp2(torch.randint(-30, 30, (R, 1), generator=g).float())
    if R > 3:
        x[1] = 0.0                      # all-zero row
        x[2, : min(C, 64)] *= 1e-30     # tiny values (subnormal codes)
        x[3, 5 % C] = 3e38              # one huge value
    return x.to(dtype)


def _host(x):
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


@pytest.mark.parametrize("mode", ["ptpc", "blockscale", "mxfp8"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C", [(1, 128), (37, 2048), (300, 7168), (5, 32768)])
def test_quantize_bit_exact(lib, mode, dtype, R, C):
    x = _make(R, C, R + C, dtype)
    q_ref, s_ref = oracle.quantize(mode, _host(x))
    q, s = lib.quantize(mode, x.cuda())
    torch.cuda.synchronize()
    q, s = q.cpu().numpy(), s.cpu().numpy()
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, [(tuple(i), hex(q[tuple(i)]), hex(q_ref[tuple(i)])) for i in bad[:5]]
    assert np.array_equal(s.view(np.uint8), s_ref.view(np.uint8))


def _near_ties(R, C, seed):
    # Every 32-column group opens with the row's amax, so every block of every
    # mode has scale s = fp32(amax / 448); the other entries are fp32(m * s)
    # moved by -6..6 ulps, m an e4m3 rounding midpoint (normal, subnormal or
    # the saturation point 464), or values whose quotient lies in the e4m3
    # subnormal band.  The quotients land on and beside the midpoints, where
    # the rounded fp32 quotient decides the code.
    rng = np.random.default_rng(seed)
    X = np.empty((R, C), np.float32)
    for r in range(R):
        amax = np.float32(np.exp2(rng.uniform(-60, 60)) * rng.uniform(1, 2))
        s = np.float32(amax / np.float32(448.0))
        e = rng.integers(-10, 9, C)
        j = rng.integers(0, 8, C)
        m = np.where(e >= -6, (1 + (2 * j + 1) / 16.0) * np.exp2(e), (2 * j + 1) * 2.0 ** -10)
        m[rng.random(C) < 0.05] = 464.0
        band = rng.random(C) < 0.1
        m[band] = np.exp2(rng.uniform(-11, -6, band.sum()))
        x = (m.astype(np.float32) * s).astype(np.float32)
        x = (x.view(np.int32) + rng.integers(-6, 7, C).astype(np.int32)).view(np.float32)
        x = np.minimum(x, amax) * np.where(rng.random(C) < 0.5, -1, 1).astype(np.float32)
        x[::32] = amax
        X[r] = x
    return X


@pytest.mark.parametrize("mode", ["ptpc", "blockscale", "mxfp8"])
@pytest.mark.parametrize("bf16", [False, True])
def test_quantize_near_rounding_midpoints(lib, mode, bf16):
    X = _near_ties(64, 1024, 11 + bf16)
    x = torch.from_numpy(X)
    if bf16:
        x = x.bfloat16()  # rounding to bf16 keeps the quotients near the midpoints of a coarser grid
    q_ref, s_ref = oracle.quantize(mode, _host(x))
    q, s = lib.quantize(mode, x.cuda())
    torch.cuda.synchronize()
    q, s = q.cpu().numpy(), s.cpu().numpy()
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, [(tuple(i), hex(q[tuple(i)]), hex(q_ref[tuple(i)])) for i in bad[:5]]
    assert np.array_equal(s.view(np.uint8), s_ref.view(np.uint8))


@pytest.mark.parametrize("mode", ["ptpc", "blockscale"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_scales_on_both_sides_of_the_reciprocal_range(lib, mode, dtype):
    # the kernel forms x / s with a reciprocal and fma corrections for scales in
    # [2^-60, 2^60] and with a division outside; rows scaled from 2^-75 to 2^70
    # put block and row scales on both sides of the bounds (and right at them)
    g = torch.Generator("cpu")
    g.manual_seed(31)
    ex = torch.tensor([-75, -69, -60, -52, -51, 0, 51, 52, 60, 61, 66, 70] * 4, dtype=torch.float32)
    x = torch.randn(ex.numel(), 2048, generator=g) * torch.exp2(ex)[:, None]
    x[::3, ::5] *= 1e-6  # small values in the same rows and blocks
    x = x.to(dtype)
    q_ref, s_ref = oracle.quantize(mode, _host(x))
    q, s = lib.quantize(mode, x.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint8), s_ref.view(np.uint8))


def test_quantize_full_size_sampled_rows(lib):
    # the largest activation of the workloads, 32768 x 7168 bf16, every mode;
    # rows are independent, so the oracle checks a sample of them
    g = torch.Generator("cpu")
    g.manual_seed(77)
    x = torch.randn(32768, 7168, generator=g).bfloat16()
    rows = np.array([0, 1, 4095, 16384, 32767] + list(np.random.default_rng(5).integers(0, 32768, 27)))
    xd = x.cuda()
    for mode in ("ptpc", "blockscale", "mxfp8"):
        q, s = lib.quantize(mode, xd)
        torch.cuda.synchronize()
        q_ref, s_ref = oracle.quantize(mode, _host(x[rows]))
        assert np.array_equal(q.cpu().numpy()[rows], q_ref), mode
        sc = s.cpu().numpy()
        sc = np.ascontiguousarray(sc[rows] if mode == "ptpc" else sc[:, rows])
        assert np.array_equal(sc.view(np.uint8), s_ref.view(np.uint8)), mode


def test_quantize_then_gemm_matches_oracle(lib):
    # GPU quantisation feeding the GPU GEMM equals the oracle's quantisation
    # feeding the oracle's GEMM
    from checker import check
    import gpu_util

    g = torch.Generator("cpu")
    g.manual_seed(8)
    a = torch.randn(256, 1024, generator=g).bfloat16()
    b = (torch.randn(512, 1024, generator=g) * 0.02).bfloat16()
    for mode in ("ptpc", "blockscale", "mxfp8"):
        qa, sa = lib.quantize(mode, a.cuda())
        if mode == "blockscale":
            import synth

            qb_c, sb_c = synth.quantize_e4m3_blocks_128x128(b.float())
            qb, sb = qb_c.cuda(), sb_c.cuda()
        else:
            qb, sb = lib.quantize(mode, b.cuda())
        C = torch.empty(256, 512, dtype=torch.bfloat16, device="cuda")
        h = lib.scaled_gemm_create(mode, 512, 1024, 256)
        lib.scaled_gemm_launch(h, qa.data_ptr(), qb.data_ptr(), sa.data_ptr(), sb.data_ptr(), C.data_ptr(), 256)
        torch.cuda.synchronize()
        lib.scaled_gemm_destroy(h)
        qa_r, sa_r = oracle.quantize(mode, _host(a))
        if mode == "blockscale":
            qb_r, sb_r = qb_c.numpy(), sb_c.numpy()
        else:
            qb_r, sb_r = oracle.quantize(mode, _host(b))
        _, ref = oracle.gemm(mode, qa_r, qb_r, sa_r, sb_r, want_r=False)
        r = check(C.view(torch.int16).cpu().numpy().view(np.uint16), ref)
        assert r["ok"], (mode, r)
