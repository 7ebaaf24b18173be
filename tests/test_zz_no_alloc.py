"""scaled_gemm_launch_noalloc: the ptpc GEMM for callers that cannot allocate
device memory (inside a custom allocator or pool callback, or when a pool owns
all device memory).  It keeps the kernel's status record in a static device
array instead of a cudaMalloc'd one.

The test calls it through the C ABI on two calls in a row (and more, into
NaN-poisoned outputs) and compares every output element by element with the
CPU oracle, within the same element-wise / relL2 tolerance as the other GPU
tests, and with the handle-based scaled_gemm_launch on the same inputs (bit
for bit, since both run the same kernel).  It is collected last so that a run
stopping at the first failure has run every other test first; it passes alone
in a fresh process too (the first call sets the device up).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = pytest.mark.gpu


# the first three shapes take the 128-wide tile (fewer 256-wide tiles than pairs
# of SMs), the last one the 256-wide tile (128 of them)
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 528, 416), (129, 144, 1152), (4096, 2048, 512)])
def test_noalloc_matches_oracle_and_handle_launch(M, N, K):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util
    from fp8_scaled_gemm_sm_gb300 import binding

    gpu_util.lib_ready()
    case = synth.make_case("ptpc", M, N, K, seed=M + N, b_std=0.02)
    _, ref = oracle.gemm("ptpc", *case.numpy(), want_r=False)
    dc = gpu_util.DeviceCase(case)
    h = gpu_util.make_plan(case)
    try:
        dc.poison()
        dc.launch(h)
        torch.cuda.synchronize()
        want = dc.c_bits()
    finally:
        binding.scaled_gemm_destroy(h)
    assert check(want, ref)["ok"]
    s = torch.cuda.current_stream().cuda_stream
    for call in range(4):
        dc.poison()
        binding.scaled_gemm_launch_noalloc(
            dc.A.data_ptr(), dc.B.data_ptr(), dc.sa.data_ptr(), dc.sb.data_ptr(), dc.C.data_ptr(), M, N, K, s
        )
        torch.cuda.synchronize()
        got = dc.c_bits()
        r = check(got, ref)
        assert r["ok"], (call, r)
        assert np.array_equal(got, want), "call %d differs from the handle launch" % call
        assert dc.canary_ok()
