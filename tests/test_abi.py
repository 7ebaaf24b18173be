"""The C-ABI library without a GPU: it loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before touching
CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from fp8_scaled_gemm_sm_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(scaled_gemm_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_header_declares_the_api():
    names = _declared()
    for n in ("scaled_gemm_create", "scaled_gemm_launch", "scaled_gemm_destroy", "scaled_gemm_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(binding.LIB_PATH)
    for n in _declared():
        assert hasattr(raw, n), n
        assert n in binding.SIGNATURES, "binding lacks " + n


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.scaled_gemm_status_string(code)
    assert "unknown" in binding.scaled_gemm_status_string(99)


@pytest.mark.parametrize(
    "mode,N,K,M_max,status",
    [
        (7, 256, 256, 16, 1),        # bad mode
        ("ptpc", -16, 256, 16, 1),   # negative size
        ("ptpc", 100, 256, 16, 2),   # N % 16
        ("ptpc", 256, 24, 16, 2),    # K % 16
        ("bf16", 256, 12, 16, 2),    # K % 8
        ("blockscale", 256, 192, 16, 2),  # K % 128
        ("mxfp8", 256, 48, 16, 2),   # K % 32
        ("ptpc", 1 << 31, 256, 16, 2),  # too large
    ],
)
def test_create_rejects_bad_shapes_on_the_host(lib, mode, N, K, M_max, status):
    with pytest.raises(binding.ScaledGemmError) as e:
        binding.scaled_gemm_create(mode, N, K, M_max)
    assert e.value.status == status


def test_null_handle_is_rejected(lib):
    L = binding.lib()
    assert L.scaled_gemm_launch(None, None, None, None, None, None, 16, None) == 1
    assert L.scaled_gemm_destroy(None) == 0
    assert L.scaled_gemm_get_config(None, None, None, None, None, None) == 1
    assert L.scaled_gemm_set_debug(None, 0, -1) == 1
    assert L.scaled_gemm_set_tile(None, 0) == 1
    code = ctypes.c_int32()
    assert L.scaled_gemm_debug_status(None, None, ctypes.byref(code), None) == 1
    assert L.scaled_gemm_create(None, 1, 256, 256, 16, -1) == 1


def test_noalloc_rejects_bad_arguments_on_the_host(lib):
    L = binding.lib()
    f = L.scaled_gemm_launch_noalloc
    assert f(None, None, None, None, None, 16, 100, 256, None) == 2   # N % 16
    assert f(None, None, None, None, None, 16, 256, 24, None) == 2    # K % 16
    assert f(None, None, None, None, None, -1, 256, 256, None) == 1   # negative
    assert f(None, None, None, None, None, 0, 256, 256, None) == 0    # empty: nothing to do
    assert f(None, None, None, None, None, 16, 256, 256, None) == 1   # NULL operands
    assert f(16, 32, 48, 64, 8, 16, 256, 256, None) == 3              # C misaligned


def test_gather_rejects_a_null_handle_on_the_host(lib):
    f = binding.lib().scaled_gemm_launch_gather
    assert f(None, None, 16, None, None, None, None, None, 16, None) == 1   # NULL handle
    # (checks on a plan -- wrong mode, bad R, NULL or misaligned operands -- need a
    # device to create the plan and run in tests/test_gpu_gather.py)


def test_quantize_rejects_bad_arguments_on_the_host(lib):
    f = binding.lib().scaled_gemm_quantize
    assert f(0, 0, None, 4, 128, None, None, None) == 1        # bf16 mode is not a quantisation mode
    assert f(1, 7, None, 4, 128, None, None, None) == 1        # bad dtype
    assert f(1, 0, None, 4, 24, None, None, None) == 2         # C % 16
    assert f(2, 0, None, 4, 64, None, None, None) == 2         # C % 128
    assert f(3, 0, None, 4, 48, None, None, None) == 2         # C % 32
    assert f(1, 0, None, 4, 65536, None, None, None) == 2      # C too large
    assert f(1, 0, None, 0, 128, None, None, None) == 0        # nothing to do
    assert f(1, 0, None, 4, 128, None, None, None) == 1        # NULL pointers
    assert f(1, 0, 16, 4, 128, 8, 32, None) == 3               # misaligned


def test_noalloc_rejects_c_overlapping_a_scale_buffer_on_the_host(lib):
    # C [16, 256] bf16 occupies 8 KB from 0x300000; any scale buffer inside it is
    # refused before the library touches the device (addresses are never dereferenced)
    f = binding.lib().scaled_gemm_launch_noalloc
    A, B, C = 0x100000, 0x200000, 0x300000
    assert f(A, B, C + 4096, 0x400000, C, 16, 256, 256, None) == 1      # a_scale inside C
    assert f(A, B, 0x400000, C + 8192 - 16, C, 16, 256, 256, None) == 1  # b_scale's first bytes inside C
    assert f(A, B, C - 32, 0x400000, C, 16, 256, 256, None) == 1         # a_scale (64 B) straddles C's start
    assert f(C, B, 0x400000, 0x500000, C, 16, 256, 256, None) == 1       # A is C
