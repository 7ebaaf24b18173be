"""GPU parity for the gather-GEMM (scaled_gemm_launch_gather through the C ABI)
against the CPU oracle: output row i is the ptpc GEMM row of source row idx[i]
(ROCm/aiter PR 6539, Technical Details: gather_kv_b_proj).

Every case is launched several times into a NaN-poisoned output with a guard
tail; launch 0 is compared with the oracle element by element, later launches
must be bit-identical to it (ROCm/aiter PR 6539, Test Plan: repeated launches
into a NaN-filled output against an fp32 reference).
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0
CANARY = 0x5A5A


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util

    gpu_util.lib_ready()
    from fp8_scaled_gemm_sm_gb300 import binding

    return binding


class GatherDev:
    def __init__(self, case, idx=None):
        self.case = case
        self.A = case.A_src.cuda()
        self.sa = case.sa_src.cuda()
        self.B = case.B.cuda()
        self.sb = case.sb.cuda()
        self.idx_host = (case.idx if idx is None else torch.as_tensor(idx, dtype=torch.int32)).contiguous()
        self.idx = self.idx_host.cuda()
        self.M = self.idx_host.numel()
        self.buf = torch.empty(self.M * case.N + 4096, dtype=torch.int16, device="cuda")
        self.C = self.buf[: self.M * case.N].view(self.M, case.N)
        self.buf[self.M * case.N:].fill_(CANARY)

    def launch(self, binding, h, R=None):
        binding.scaled_gemm_launch_gather(
            h, self.A.data_ptr(), self.case.R if R is None else R, self.idx.data_ptr(), self.B.data_ptr(),
            self.sa.data_ptr(), self.sb.data_ptr(), self.C.data_ptr(), self.M,
            torch.cuda.current_stream().cuda_stream)

    def bits(self):
        return self.C.cpu().numpy().view(np.uint16)

    def canary_ok(self):
        return bool((self.buf[self.M * self.case.N:] == CANARY).all().item())


def _run(binding, case, idx=None, launches=8, ms=None, ns=None):
    d = GatherDev(case, idx)
    A, _, B, sa, sb = case.numpy()
    idx_np = d.idx_host.numpy()
    if ms is None:
        _, ref = oracle.gemm_gather(A, idx_np, B, sa, sb, want_r=False)
    else:
        _, ref = oracle.gemm_gather_points(A, idx_np, B, sa, sb, ms, ns)
    h = binding.scaled_gemm_create("ptpc", case.N, case.K, d.M)
    try:
        first = None
        for i in range(launches):
            d.C.fill_(NAN_BF16)
            d.launch(binding, h)
            torch.cuda.synchronize()
            assert not bool(torch.isnan(d.C.view(torch.bfloat16)).any()), "NaN in launch %d" % i
            if first is None:
                first = d.C.clone()
                got = d.bits() if ms is None else d.bits()[ms, ns]
                r = check(got, ref)
                assert r["ok"], r
            else:
                assert torch.equal(d.C, first), "launch %d differs from launch 0" % i
            assert d.canary_ok()
        code, where = binding.scaled_gemm_debug_status(h)
        assert code == 0, (code, where)
    finally:
        binding.scaled_gemm_destroy(h)
    return first


@pytest.mark.parametrize(
    "M,R,N,K",
    [
        (1, 64, 16, 32),          # one row, one partial K block
        (130, 4096, 528, 512),    # ragged M and N, the workload's K
        (513, 8192, 1168, 256),   # tail-only K (two blocks), ragged everything
        (256, 2048, 256, 2048),   # long K (16 blocks)
        (200, 1024, 8192, 512),   # the workload's N
    ],
)
def test_gather_shapes(lib, M, R, N, K):
    _run(lib, synth.make_gather_case(M, R, N, K, seed=M + K, page=16))


def test_gather_out_of_range_and_repeated_indices(lib):
    case = synth.make_gather_case(160, 300, 272, 512, seed=3, page=16)
    rng = np.random.default_rng(4)
    idx = rng.integers(0, 300, 160).astype(np.int64)
    idx[::7] = -1
    idx[3::11] = 300
    idx[5::13] = 2**31 - 1
    idx[10:20] = 42
    C = _run(lib, case, idx=idx.astype(np.int32))
    bad = (idx < 0) | (idx >= 300)
    c = C.view(torch.bfloat16).float().cpu().numpy()
    assert np.all(c[bad] == 0.0)
    assert np.array_equal(c[10], c[19])


def test_identity_gather_equals_the_plain_launch_bit_for_bit(lib):
    # the gather kernel (one CTA per 128 x 256 tile) and the plain launch (the pair
    # kernel) sum every element over K in the same order of K = 32 MMA steps and
    # apply the scales alike, so the outputs agree bitwise
    import gpu_util

    plain = synth.make_case("ptpc", 384, 512, 512, seed=9, b_std=0.02)
    g = synth.GatherCase(384, 512, 512, 384, plain.A, plain.sa, torch.arange(384, dtype=torch.int32),
                         plain.B, plain.sb)
    Cg = _run(lib, g, launches=2)
    dc = gpu_util.DeviceCase(plain)
    h = gpu_util.make_plan(plain)
    try:
        dc.poison()
        dc.launch(h)
        torch.cuda.synchronize()
        assert torch.equal(dc.C, Cg.view(torch.int16).view(dc.C.shape))
    finally:
        lib.scaled_gemm_destroy(h)


def test_gather_rejections_on_a_plan(lib):
    case = synth.make_gather_case(64, 256, 256, 512, seed=5, page=16)
    d = GatherDev(case)
    h = lib.scaled_gemm_create("ptpc", 256, 512, 64)
    hb = lib.scaled_gemm_create("bf16", 256, 512, 64)
    L = lib.lib()
    s = torch.cuda.current_stream().cuda_stream
    a = (d.A.data_ptr(), 256, d.idx.data_ptr(), d.B.data_ptr(), d.sa.data_ptr(), d.sb.data_ptr(), d.C.data_ptr(), 64, s)
    try:
        assert L.scaled_gemm_launch_gather(hb, *a) == 1                                   # not a ptpc plan
        assert L.scaled_gemm_launch_gather(h, a[0], -1, *a[2:]) == 1                      # negative R
        assert L.scaled_gemm_launch_gather(h, a[0], 2**31, *a[2:]) == 2                   # R too large
        assert L.scaled_gemm_launch_gather(h, *a[:2], None, *a[3:]) == 1                  # NULL idx
        assert L.scaled_gemm_launch_gather(h, a[0] + 8, *a[1:]) == 3                      # misaligned A_src
        assert L.scaled_gemm_launch_gather(h, *a[:7], 65, s) == 1                         # M > M_max
        # no source row: every output row is zero
        d.C.fill_(NAN_BF16)
        assert L.scaled_gemm_launch_gather(h, a[0], 0, *a[2:]) == 0
        torch.cuda.synchronize()
        assert bool((d.C == 0).all())
    finally:
        lib.scaled_gemm_destroy(h)
        lib.scaled_gemm_destroy(hb)


def test_gather_skipped_stage_times_out_and_context_survives(lib):
    case = synth.make_gather_case(256, 2048, 512, 1024, seed=6, page=16)
    d = GatherDev(case)
    A, idx, B, sa, sb = case.numpy()
    _, ref = oracle.gemm_gather(A, idx, B, sa, sb, want_r=False)
    h = lib.scaled_gemm_create("ptpc", case.N, case.K, case.M)
    try:
        lib.scaled_gemm_set_debug(h, 50_000_000, 1)
        d.C.fill_(NAN_BF16)
        t0 = time.time()
        d.launch(lib, h)
        torch.cuda.synchronize()
        assert time.time() - t0 < 5.0
        code, where = lib.scaled_gemm_debug_status(h)
        assert code == 6 and where != 0, (code, where)
        lib.scaled_gemm_set_debug(h, 0, -1)
        d.C.fill_(NAN_BF16)
        d.launch(lib, h)
        torch.cuda.synchronize()
        assert check(d.bits(), ref)["ok"]
        assert lib.scaled_gemm_debug_status(h)[0] == 0
    finally:
        lib.scaled_gemm_destroy(h)


@pytest.mark.slow
def test_gather_full_size_workload(lib):
    # 16384 rows gathered from a 65536-row paged cache, N = 8192, K = 512;
    # 20 launches, oracle at sampled positions (whole rows first / middle / last,
    # the last N tile for 64 rows, 4096 random positions)
    name = "g_ptpc_gather_16384x8192x512"
    M, R, N, K, seed = synth.GATHER_CONFIGS[name]
    case = synth.make_gather_case(M, R, N, K, seed=seed)
    rng = np.random.default_rng(11)
    ms, ns = [], []
    for r in (0, M // 2 + 37, M - 1):
        ms += [r] * N
        ns += list(range(N))
    for r in rng.choice(M, 64, replace=False):
        ms += [int(r)] * 256
        ns += list(range(N - 256, N))
    ms += list(rng.integers(0, M, 4096))
    ns += list(rng.integers(0, N, 4096))
    _run(lib, case, launches=20, ms=np.array(ms), ns=np.array(ns))
