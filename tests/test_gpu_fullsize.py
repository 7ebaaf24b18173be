"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (one plan per workload, M_max = M, persistent grid).

Each workload is launched 20 times into a NaN-poisoned output with a guard
tail (ROCm/mori PR 785, Test; ROCm/aiter PR 6539, Test Plan).  Launch 0 is
compared with the CPU oracle element by element at sampled positions: three
whole rows (first, middle, last -- the last one in the ragged last M tile),
every column of the last (possibly partial) N tile for 64 rows, and 4096
random positions; rms(ref) for the tolerance is taken over that sample.  Every
later launch must be bit-identical to launch 0 (deepseek-ai/DeepGEMM PR 453,
test_bf16_repeatability), NaN-free, and leave the guard tail intact.  The
BF16 workload is repeated 1000 times.  One workload also runs with a copy loop
on a second stream of the same GPU (ROCm/mori PR 785 review: "idle and with a
copy loop on the same GPU").
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

_CACHE = {}


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util

    gpu_util.lib_ready()
    return gpu_util


def _case(name):
    mode, M, N, K, seed, a_std, b_std = synth.CONFIGS[name]
    return synth.make_case(mode, M, N, K, seed=seed, a_std=a_std, b_std=b_std, cache=_CACHE)


def _sample(case, rng):
    M, N = case.M, case.N
    ms, ns = [], []
    for r in (0, M // 2 + 37 if M > 80 else M // 2, M - 1):
        ms += [r] * N
        ns += list(range(N))
    bn_last = (N - 1) // 224 * 224 if case.mode == "mxfp8" else (N - 1) // 256 * 256
    rows = rng.choice(M, size=min(64, M), replace=False)
    for r in rows:
        ms += [int(r)] * (N - bn_last)
        ns += list(range(bn_last, N))
    ms += list(rng.integers(0, M, 4096))
    ns += list(rng.integers(0, N, 4096))
    return np.array(ms, dtype=np.int64), np.array(ns, dtype=np.int64)


def _run(gpu, name, launches=20, stress=False):
    case = _case(name)
    rng = np.random.default_rng(1234)
    ms, ns = _sample(case, rng)
    _, ref = oracle.gemm_points(case.mode, *case.numpy(), ms, ns)
    dc = gpu.DeviceCase(case)
    h = gpu.make_plan(case)
    side = None
    if stress:
        side = torch.cuda.Stream()
        src = torch.empty(256 << 20, dtype=torch.int32, device="cuda")
        dst = torch.empty_like(src)
    try:
        first = None
        for i in range(launches):
            dc.poison()
            if side is not None:
                with torch.cuda.stream(side):
                    for _ in range(4):
                        dst.copy_(src)
            dc.launch(h)
            torch.cuda.current_stream().synchronize()
            C = dc.C
            assert not bool(torch.isnan(C.view(torch.bfloat16)).any()), "NaN in launch %d" % i
            if first is None:
                first = C.clone()
                got = first.view(torch.int16).cpu().numpy().view(np.uint16)[ms, ns]
                r = check(got, ref)
                assert r["ok"], r
            else:
                assert torch.equal(C, first), "launch %d differs from launch 0" % i
            assert dc.canary_ok(), "guard tail after C was written"
        torch.cuda.synchronize()
        code, where = gpu.binding.scaled_gemm_debug_status(h)
        assert code == 0, (code, where)
    finally:
        gpu.binding.scaled_gemm_destroy(h)
        del dc
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", [k for k in synth.SUITE if not k.startswith("c4_bf16")] + ["c0_ptpc_256x512x256"])
def test_fullsize_workload(gpu, name):
    _run(gpu, name)


@pytest.mark.parametrize("name", synth.EXTRA)
def test_fullsize_extra_shape(gpu, name):
    _run(gpu, name)


def test_fullsize_bf16_1000_launches_bit_identical(gpu):
    _run(gpu, "c4_bf16_4096x896x1024", launches=1000)


def test_fullsize_under_concurrent_copy_loop(gpu):
    _run(gpu, "c2_ptpc_32768x7168x1792", launches=20, stress=True)
