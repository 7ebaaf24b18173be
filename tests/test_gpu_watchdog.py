"""The kernels' bounded waits, exercised on the GPU without faulting it.

Every mbarrier wait in the kernels gives up after a time limit, records a
timeout and the wait site in the plan's status word, lets its own copies and
MMAs in flight finish, frees its TMEM and returns.  Here the producer of every
CTA is told to skip one pipeline stage (a barrier that nothing will complete),
with a 50 ms limit: the launch must end by itself, report SG_ERR_TIMEOUT
through scaled_gemm_debug_status, and leave the context usable -- the next
launch with the skip removed must match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from checker import check

pytestmark = pytest.mark.gpu

TIMEOUT = 6


# (mode, M, N, K, pinned tile width or 0): at these M the launches choose the
# 128-wide tiles, so the wide kernels (mxfp8 224, dense 256) are pinned in cases
# of their own
@pytest.mark.parametrize("mode,M,N,K,tile", [("ptpc", 512, 512, 1024, 0), ("ptpc", 512, 512, 1024, 256),
                                             ("mxfp8", 256, 448, 1024, 0), ("mxfp8", 256, 448, 1024, 224),
                                             ("blockscale", 256, 256, 1024, 0), ("bf16", 256, 512, 512, 0),
                                             ("bf16", 256, 512, 512, 256)])
def test_skipped_stage_times_out_and_context_survives(mode, M, N, K, tile):
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    import gpu_util
    from fp8_scaled_gemm_sm_gb300 import binding

    gpu_util.lib_ready()
    case = synth.make_case(mode, M, N, K, seed=5, b_std=0.02)
    _, ref = oracle.gemm(mode, *case.numpy(), want_r=False)
    dc = gpu_util.DeviceCase(case)
    h = gpu_util.make_plan(case)
    try:
        if tile:
            binding.scaled_gemm_set_tile(h, tile)
        binding.scaled_gemm_set_debug(h, 50_000_000, 1)
        dc.poison()
        t0 = time.time()
        dc.launch(h)
        torch.cuda.synchronize()
        dt = time.time() - t0
        code, where = binding.scaled_gemm_debug_status(h)
        assert code == TIMEOUT, (code, where)
        assert where != 0
        assert dt < 5.0, dt
        # the context is still usable and the next launch is correct
        binding.scaled_gemm_set_debug(h, 0, -1)
        dc.poison()
        dc.launch(h)
        torch.cuda.synchronize()
        assert check(dc.c_bits(), ref)["ok"]
        code, _ = binding.scaled_gemm_debug_status(h)
        assert code == 0
    finally:
        binding.scaled_gemm_destroy(h)
