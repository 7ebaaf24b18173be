"""GPU parity on the edge matrices of every kernel family, through the C ABI,
against the CPU oracle element by element.

Each case is launched 8 times into a NaN-poisoned output with a guard tail;
every launch must pass the element-wise and relL2 bounds, be NaN-free, be
bit-identical to the first and leave the guard tail intact (ROCm/mori PR 785,
Test; ROCm/aiter PR 6539, Test Plan).

* The pair kernel (ptpc and bf16, 256- and 128-wide tiles) at one-row, ragged
  and tile-sized M against N of 16, 48 and 144 columns: the odd CTA of a pair
  tile wholly past M, and a CTA's half of B wholly past N (ROCm/mori PR 809,
  Worth a reviewer's attention: the partial last column tile), at K of 5 and 9
  blocks.
* The short-K matrix: K of one to four 128-wide blocks (and one to eight
  64-wide bf16 blocks), including the tail-only K <= 256 where the K loop is
  all tail (ROCm/mori PR 785, Problem), at N = 16, 144 and 6288, both widths.
* mxfp8 with e8m0 scale codes 0, 1, 127, 253 and 254 mixed per K block (ROCm/mori
  PR 785, cost table and Scope: the mode's power-of-two block scales).
* blockscale with fp32 scales spread over 2^-40 .. 2^40, some of them zero.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util

    gpu_util.lib_ready()
    return gpu_util


def _run(gpu, case, launches=8, tile_bn=0):
    _, ref = oracle.gemm(case.mode, *case.numpy(), want_r=False)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    try:
        if tile_bn:
            gpu.binding.scaled_gemm_set_tile(h, tile_bn)
        first = None
        for i in range(launches):
            dc.poison()
            dc.launch(h)
            torch.cuda.synchronize()
            bits = dc.c_bits()
            r = check(bits, ref)
            assert r["ok"], (i, r)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), "launch %d differs from launch 0" % i
            assert dc.canary_ok(), "guard tail after C was written"
        code, where = gpu.binding.scaled_gemm_debug_status(h)
        assert code == 0, (code, where)
    finally:
        gpu.binding.scaled_gemm_destroy(h)
    return first, ref


# these shapes have fewer 256-wide tiles than pairs of SMs, so a launch left to
# choose takes the 128-wide tile: both widths are pinned in turn
@pytest.mark.parametrize("tile", [128, 256])
@pytest.mark.parametrize("mode", ["ptpc", "bf16"])
@pytest.mark.parametrize("K", [640, 1152])
@pytest.mark.parametrize("N", [16, 48, 144])
@pytest.mark.parametrize("M", [1, 127, 129])
def test_pair_kernel_edges(gpu, mode, M, N, K, tile):
    b_std = 0.02 if mode == "ptpc" else 1.0
    _run(gpu, synth.make_case(mode, M, N, K, seed=M * 7 + N + K, b_std=b_std), tile_bn=tile)


@pytest.mark.parametrize("tile", [128, 256])
@pytest.mark.parametrize("mode", ["ptpc", "bf16"])
@pytest.mark.parametrize("N", [16, 144, 6288])
@pytest.mark.parametrize("K", [32, 64, 128, 256, 384, 512])
def test_short_k_matrix(gpu, mode, K, N, tile):
    b_std = 0.02 if mode == "ptpc" else 1.0
    _run(gpu, synth.make_case(mode, 129, N, K, seed=K + N, b_std=b_std), tile_bn=tile)


@pytest.mark.parametrize("M,N,K,tile", [(256, 448, 1024, 224), (300, 672, 2080, 224), (256, 448, 1024, 128),
                                        (383, 7168, 256, 0)])
def test_mxfp8_extreme_scale_codes(gpu, M, N, K, tile):
    base = synth.make_case("mxfp8", M, N, K, seed=M + K, b_std=0.02)
    case = synth.with_extreme_mx_codes(base, seed=K)
    got_codes = set(np.unique(case.sa.numpy())) | set(np.unique(case.sb.numpy()))
    assert {0, 1, 253, 254} <= got_codes
    _, ref = oracle.gemm("mxfp8", *case.numpy(), want_r=False)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    try:
        if tile:
            gpu.binding.scaled_gemm_set_tile(h, tile)
        first = None
        for i in range(8):
            dc.poison()
            dc.launch(h)
            torch.cuda.synchronize()
            bits = dc.c_bits()
            r = check(bits, ref)
            assert r["ok"], (i, r)
            first = bits if first is None else first
            assert np.array_equal(bits, first)
            assert dc.canary_ok()
    finally:
        gpu.binding.scaled_gemm_destroy(h)


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (383, 896, 1152), (129, 144, 2048)])
def test_blockscale_wide_and_zero_scales(gpu, M, N, K):
    base = synth.make_case("blockscale", M, N, K, seed=M + N, b_std=0.02)
    case = synth.with_wide_block_scales(base, seed=M)
    got, _ = _run(gpu, case)
    # the A row whose block scales are all zero comes out zero
    assert np.all((got.reshape(M, N)[M // 2] & 0x7FFF) == 0)


def test_launch_rejects_c_overlapping_a_scale_buffer(gpu):
    # C must not overlap a scale buffer: the launch is refused on the host
    case = synth.make_case("ptpc", 64, 256, 256, seed=2)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    L = gpu.binding.lib()
    s = torch.cuda.current_stream().cuda_stream
    try:
        c = dc.C.data_ptr()
        assert L.scaled_gemm_launch(h, dc.A.data_ptr(), dc.B.data_ptr(), c + 256, dc.sb.data_ptr(), c, 64, s) == 1
        assert L.scaled_gemm_launch(h, dc.A.data_ptr(), dc.B.data_ptr(), dc.sa.data_ptr(), c, c, 64, s) == 1
        hb = gpu.binding.scaled_gemm_create("blockscale", 256, 256, 64)
        try:
            # blockscale a_scale is [K/128][M] fp32 = 512 bytes: ending 16 bytes into C overlaps
            assert L.scaled_gemm_launch(hb, dc.A.data_ptr(), dc.B.data_ptr(), c - 512 + 16, dc.sb.data_ptr(), c, 64, s) == 1
        finally:
            gpu.binding.scaled_gemm_destroy(hb)
    finally:
        gpu.binding.scaled_gemm_destroy(h)
