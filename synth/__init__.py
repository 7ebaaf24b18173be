"""Seeded synthetic inputs for the scaled FP8 / BF16 GEMM.

This package is shared by the tests, the benchmark and the smoke check.  It
holds input preparation only -- random draws and the per-row / per-block
quantisation that turns them into e4m3 codes plus scales -- and none of the
GEMM arithmetic.  Both the CUDA path and the CPU oracle read the same bytes
it produces.
"""
from .gen import (  # noqa: F401
    Case,
    SUITE,
    EXTRA,
    CONFIGS,
    make_case,
    GatherCase,
    make_gather_case,
    paged_indices,
    GATHER_CONFIGS,
    make_int_case,
    with_extreme_mx_codes,
    with_wide_block_scales,
    quantize_e4m3_rows,
    quantize_e4m3_blocks_1x128,
    quantize_e4m3_blocks_128x128,
    quantize_mx_rows,
    gemm_flops,
    gemm_bytes,
)
