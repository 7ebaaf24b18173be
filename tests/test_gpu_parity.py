"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle, element by element, on NaN-poisoned outputs with a guard tail.

Every case is launched repeatedly (20 times unless stated) and every launch
must (i) pass the element-wise bound |c - ref| <= 0.02|ref| + 0.01 rms(ref) and
relL2 <= 3e-3, (ii) contain no NaN, (iii) be bit-identical to the first launch
and (iv) leave the guard tail after C untouched.  Repeated launches into a
poisoned output are the protocol of ROCm/mori PR 785 (Test) and ROCm/aiter PR
6539 (Test Plan); bit-identity across launches is deepseek-ai/DeepGEMM PR 453
(test_bf16_repeatability).
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


def _run_full(gpu, case, launches=20, tile_bn=0):
    """Full comparison against the oracle on every launch (`tile_bn`: the plan's
    pinned output-tile width, 0 = chosen per launch)."""
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


def test_config0_ptpc_256x512x256(gpu):
    _run_full(gpu, synth.make_case("ptpc", 256, 512, 256, seed=0))


@pytest.mark.parametrize(
    "M,N,K",
    [
        (1, 16, 16),        # smallest legal problem
        (127, 48, 128),     # one K block: the main loop never runs
        (128, 256, 256),    # exactly one tile, two K blocks
        (129, 144, 256),    # ragged M and N
        (300, 528, 416),    # several tiles, ragged K (last block 32 wide)
        (513, 1168, 1792),  # partial last N tile (N = 1168), 14 K blocks
    ],
)
def test_ptpc_shapes(gpu, M, N, K):
    _run_full(gpu, synth.make_case("ptpc", M, N, K, seed=M + N, b_std=0.02), launches=8)


def test_ptpc_integer_operands_bit_exact(gpu):
    # Integer-valued operands, unit scales: sums are exact in fp32 (< 2^24), so
    # the GPU's bf16 must equal the oracle's bit for bit.  This also pins the
    # tensor core's accumulator to full fp32 precision over K = 4096.
    case = synth.make_int_case(256, 512, 4096, -16, 16, seed=3)
    got, ref = _run_full(gpu, case, launches=4)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 528, 1032), (512, 896, 1024)])
def test_bf16_shapes(gpu, M, N, K):
    _run_full(gpu, synth.make_case("bf16", M, N, K, seed=233), launches=8)


def test_k_zero_writes_zero(gpu):
    case = synth.make_case("ptpc", 64, 32, 16, seed=1)
    dc = gpu.DeviceCase(case)
    h = gpu.binding.scaled_gemm_create("ptpc", 32, 0, 64)
    try:
        dc.poison()
        gpu.binding.scaled_gemm_launch(h, 0, 0, 0, 0, dc.C.data_ptr(), 64)
        torch.cuda.synchronize()
        assert np.all(dc.c_bits() == 0)
    finally:
        gpu.binding.scaled_gemm_destroy(h)


def test_m_zero_is_a_no_op(gpu):
    case = synth.make_case("ptpc", 16, 32, 32, seed=1)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    try:
        dc.poison()
        dc.launch(h, M=0)
        torch.cuda.synchronize()
        assert np.all(dc.c_bits() == gpu.NAN_BF16)
    finally:
        gpu.binding.scaled_gemm_destroy(h)


@pytest.mark.parametrize(
    "M,N,K",
    [
        (16, 16, 32),       # one partial K block (1 of 4 scale blocks)
        (1, 16, 64),        # one row: the pair's second CTA reads only zero-filled rows
        (128, 224, 128),    # one tile
        (144, 240, 416),    # ragged M, N and K (K = 3.25 stages)
        (256, 512, 1792),
        (384, 7168, 256),   # the full weight width, two K blocks
        (200, 448, 1024),   # M not a multiple of 16
        (383, 672, 2080),   # odd number of 128-row chunks, ragged last K step (65 scale blocks)
    ],
)
def test_mxfp8_shapes(gpu, M, N, K):
    _run_full(gpu, synth.make_case("mxfp8", M, N, K, seed=M + K, b_std=0.02), launches=8)


@pytest.mark.parametrize(
    "M,N,K",
    [
        (1, 16, 128),
        (128, 128, 256),
        (200, 272, 640),    # ragged M and N (N block partially outside)
        (256, 512, 2048),
        (384, 896, 1152),   # the odd CTA of a pair tile wholly past M, its B half wholly past N; 9 K blocks
        (2304, 2304, 384),  # 81 pair tiles on 76 pairs: second tiles, the partial ring's parity across tiles
    ],
)
def test_blockscale_shapes(gpu, M, N, K):
    _run_full(gpu, synth.make_case("blockscale", M, N, K, seed=M + K, b_std=0.02), launches=8)


@pytest.mark.parametrize(
    "M,N,K",
    [
        (1, 16, 32),         # one row, 16 of a tile's 128 columns, one K block of 32
        (200, 448, 1024),    # ragged M, 3.5 tiles of 128 columns
        (383, 672, 2080),    # odd number of 128-row chunks, partial last tile, ragged last K step
        (256, 7168, 1792),   # the workload's N and K at one pair row (the automatic choice is narrow)
        (2304, 1280, 384),   # 90 pair tiles on 76 pairs: second tiles, both accumulators
    ],
)
def test_mxfp8_narrow_tiles(gpu, M, N, K):
    # 256 x 128 pair tiles: B staged 64 rows per CTA, B's scales in 512-byte records
    _run_full(gpu, synth.make_case("mxfp8", M, N, K, seed=M + K + 1, b_std=0.02), launches=8, tile_bn=128)


@pytest.mark.parametrize(
    "mode,M,N,K",
    [
        ("ptpc", 1, 16, 16),        # smallest legal problem
        ("ptpc", 129, 144, 1152),   # ragged M and N, 9 K blocks
        ("ptpc", 300, 528, 416),    # several tiles, ragged K, half-tile N tail (528 = 4 x 128 + 16)
        ("ptpc", 2304, 1280, 384),  # 90 pair tiles on 76 pairs: second tiles, both accumulators
        ("bf16", 200, 448, 1024),   # ragged M, 3.5 tiles of 128 columns
        ("bf16", 513, 1168, 320),   # partial last tile, ragged bf16 K (5 blocks of 64)
    ],
)
def test_dense_narrow_tiles(gpu, mode, M, N, K):
    # 256 x 128 pair tiles: B staged 64 rows per CTA, 32 columns per epilogue
    # warp, 7 stages; the MMAs sum each output element over K in the same order
    # as on the 256-wide tile, so the two widths agree bit for bit
    case = synth.make_case(mode, M, N, K, seed=M + N + K, b_std=0.02 if mode == "ptpc" else 1.0)
    narrow, _ = _run_full(gpu, case, launches=8, tile_bn=128)
    wide, _ = _run_full(gpu, case, launches=2, tile_bn=256)
    assert np.array_equal(narrow, wide)


def test_dense_tile_width_follows_m(gpu):
    # 128-wide where 256-wide tiles would not fill the pairs of SMs (one pair row
    # of 28 tiles at M = 256), 256-wide otherwise; set_tile pins or restores
    b = gpu.binding
    small = b.scaled_gemm_create("ptpc", 7168, 7168, 256)
    large = b.scaled_gemm_create("ptpc", 7168, 7168, 4096)
    bf = b.scaled_gemm_create("bf16", 896, 1024, 4096)
    try:
        assert b.scaled_gemm_get_config(small)["bn"] == 128
        assert b.scaled_gemm_get_config(small)["stages"] == 7
        assert b.scaled_gemm_get_config(large)["bn"] == 256
        assert b.scaled_gemm_get_config(bf)["bn"] == 256  # 64 wide tiles: one wave either way
        b.scaled_gemm_set_tile(large, 128)
        assert b.scaled_gemm_get_config(large)["bn"] == 128
        b.scaled_gemm_set_tile(large, 0)
        assert b.scaled_gemm_get_config(large)["bn"] == 256
    finally:
        for h in (small, large, bf):
            b.scaled_gemm_destroy(h)


def test_dense_plan_switches_width_between_launches(gpu):
    # one plan launched back to back with an M that takes the 128-wide tile (256
    # rows: 8 wide tiles for 76 pairs) and one that takes the 256-wide tile (4096
    # rows): every launch matches the oracle on its rows and leaves the rows past
    # its M untouched
    case = synth.make_case("ptpc", 4096, 2048, 512, seed=51, b_std=0.02)
    _, ref = oracle.gemm("ptpc", *case.numpy(), want_r=False)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    try:
        for M in (256, 4096, 256, 4096):
            dc.poison()
            dc.launch(h, M=M)
            torch.cuda.synchronize()
            bits = dc.c_bits()
            r = check(bits[:M], ref[:M])
            assert r["ok"], (M, r)
            assert (bits[M:] == gpu.NAN_BF16).all(), "rows past M were written (M = %d)" % M
            assert dc.canary_ok()
        code, where = gpu.binding.scaled_gemm_debug_status(h)
        assert code == 0, (code, where)
    finally:
        gpu.binding.scaled_gemm_destroy(h)


def test_mxfp8_tile_width_follows_m(gpu):
    # a plan reports the width of a launch at M_max: 128 where 224-wide tiles would
    # leave pairs of SMs idle, 224 otherwise; set_tile pins a width or restores the choice
    b = gpu.binding
    small = b.scaled_gemm_create("mxfp8", 7168, 1792, 256)
    large = b.scaled_gemm_create("mxfp8", 7168, 1792, 32768)
    dense = b.scaled_gemm_create("ptpc", 7168, 1792, 256)
    try:
        assert b.scaled_gemm_get_config(small)["bn"] == 128
        assert b.scaled_gemm_get_config(large)["bn"] == 224
        b.scaled_gemm_set_tile(large, 128)
        assert b.scaled_gemm_get_config(large)["bn"] == 128
        b.scaled_gemm_set_tile(large, 0)
        assert b.scaled_gemm_get_config(large)["bn"] == 224
        L = b.lib()
        assert L.scaled_gemm_set_tile(large, 256) == 1 and L.scaled_gemm_set_tile(large, 96) == 1
        assert L.scaled_gemm_set_tile(dense, 224) == 1 and L.scaled_gemm_set_tile(dense, 96) == 1
        assert L.scaled_gemm_set_tile(dense, 128) == 0 and L.scaled_gemm_set_tile(dense, 256) == 0
    finally:
        for h in (small, large, dense):
            b.scaled_gemm_destroy(h)
    from fp8_scaled_gemm_sm_gb300 import ScaledGemm

    op = ScaledGemm("mxfp8", 7168, 1792, 32768)
    try:
        assert op.config()["bn"] == 224
        op.set_tile(128)
        assert op.config()["bn"] == 128
        op.set_tile()
        assert op.config()["bn"] == 224
    finally:
        op.close()


def test_mxfp8_back_to_back_launches_on_one_plan(gpu):
    # an mxfp8 plan rearranges each launch's scales in its workspace: two
    # launches with different operands queued on one stream, with no host
    # synchronisation between them, must each match their own oracle result
    c1 = synth.make_case("mxfp8", 384, 448, 1024, seed=21, b_std=0.02)
    c2 = synth.make_case("mxfp8", 384, 448, 1024, seed=22, b_std=0.02)
    _, r1 = oracle.gemm("mxfp8", *c1.numpy(), want_r=False)
    _, r2 = oracle.gemm("mxfp8", *c2.numpy(), want_r=False)
    d1, d2 = gpu.DeviceCase(c1), gpu.DeviceCase(c2)
    h = gpu.make_plan(c1)
    try:
        d1.poison()
        d2.poison()
        for _ in range(3):
            d1.launch(h)
            d2.launch(h)
        torch.cuda.synchronize()
        assert check(d1.c_bits(), r1)["ok"]
        assert check(d2.c_bits(), r2)["ok"]
        assert d1.canary_ok() and d2.canary_ok()
    finally:
        gpu.binding.scaled_gemm_destroy(h)
