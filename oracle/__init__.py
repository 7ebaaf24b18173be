"""CPU oracle for the scaled FP8 / BF16 GEMM -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline and
reference arms may import this package.  It wraps ``oracle.c`` (plain C,
binary64 accumulation, exact e4m3 / e8m0 / bf16 decoders) through ctypes and
shares no code with the CUDA library.  See oracle.c for the definition it
computes and the passages it follows.

Array conventions (numpy, C-contiguous):
  A  [M, K] uint8 e4m3fn codes (uint16 bf16 bits in bf16 mode)
  B  [N, K] same type as A
  ptpc        sa float32 [M],        sb float32 [N]
  blockscale  sa float32 [K/128, M], sb float32 [ceil(N/128), K/128]
  mxfp8       sa uint8   [K/32, M],  sb uint8   [K/32, N]   (e8m0 codes)
  bf16        sa = sb = None
"""
import ctypes
import os

import numpy as np

from . import build as _build

MODES = {"bf16": 0, "ptpc": 1, "blockscale": 2, "mxfp8": 3}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.sgo_dec_e4m3.restype = ctypes.c_double
        L.sgo_dec_e4m3.argtypes = [ctypes.c_uint8]
        L.sgo_dec_e8m0.restype = ctypes.c_double
        L.sgo_dec_e8m0.argtypes = [ctypes.c_uint8]
        L.sgo_dec_bf16.restype = ctypes.c_double
        L.sgo_dec_bf16.argtypes = [ctypes.c_uint16]
        L.sgo_bf16_rne.restype = ctypes.c_uint16
        L.sgo_bf16_rne.argtypes = [ctypes.c_double]
        i64 = ctypes.c_int64
        vp = ctypes.c_void_p
        L.sgo_gemm_rows.restype = ctypes.c_int
        L.sgo_gemm_rows.argtypes = [ctypes.c_int, i64, i64, i64, vp, vp, vp, vp, i64, i64, vp, vp]
        L.sgo_gemm_points.restype = ctypes.c_int
        L.sgo_gemm_points.argtypes = [ctypes.c_int, i64, i64, i64, vp, vp, vp, vp, i64, vp, vp, vp, vp]
        L.sgo_num_threads.restype = ctypes.c_int
        L.sgo_num_threads.argtypes = []
        L.sgo_e4m3_rne_sat.restype = ctypes.c_uint8
        L.sgo_e4m3_rne_sat.argtypes = [ctypes.c_double]
        L.sgo_quantize.restype = ctypes.c_int
        L.sgo_quantize.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, vp, vp, vp]
        _lib = L
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle's GEMM loops use."""
    return int(lib().sgo_num_threads())


def dec_e4m3(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.sgo_dec_e4m3(int(b)) for b in c.ravel()], dtype=np.float64).reshape(c.shape)


def dec_e8m0(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.sgo_dec_e8m0(int(b)) for b in c.ravel()], dtype=np.float64).reshape(c.shape)


def dec_bf16(bits) -> np.ndarray:
    L = lib()
    c = np.asarray(bits, dtype=np.uint16)
    return np.array([L.sgo_dec_bf16(int(b)) for b in c.ravel()], dtype=np.float64).reshape(c.shape)


def bf16_rne(x) -> np.ndarray:
    """Round binary64 values to bf16 bits (uint16), nearest-even, in one step."""
    L = lib()
    v = np.asarray(x, dtype=np.float64)
    return np.array([L.sgo_bf16_rne(float(t)) for t in v.ravel()], dtype=np.uint16).reshape(v.shape)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(mode, A, B, sa, sb):
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    dt = np.uint16 if m == 0 else np.uint8
    A = np.ascontiguousarray(A).view(dt)
    B = np.ascontiguousarray(B).view(dt)
    if m == 0:
        sa = sb = None
    elif m == 3:
        sa = np.ascontiguousarray(sa, dtype=np.uint8)
        sb = np.ascontiguousarray(sb, dtype=np.uint8)
    else:
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        sb = np.ascontiguousarray(sb, dtype=np.float32)
    return m, A, B, sa, sb


def gemm(mode, A, B, sa, sb, rows=None, want_r=True):
    """Rows ``rows=(m0, m1)`` (default all) of the result.

    Returns ``(R, ref)``: R float64 [rows, N] (None unless ``want_r``) and
    ref uint16 bf16 bits [rows, N].
    """
    m, A, B, sa, sb = _prep(mode, A, B, sa, sb)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    m0, m1 = (0, M) if rows is None else rows
    R = np.empty((m1 - m0, N), dtype=np.float64) if want_r else None
    ref = np.empty((m1 - m0, N), dtype=np.uint16)
    rc = lib().sgo_gemm_rows(m, M, N, K, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), m0, m1, _ptr(R), _ptr(ref))
    if rc != 0:
        raise ValueError("oracle gemm rejected its arguments (rc=%d)" % rc)
    return R, ref


def gemm_points(mode, A, B, sa, sb, ms, ns):
    """Elements (ms[i], ns[i]) computed one by one: returns (R float64, ref uint16)."""
    m, A, B, sa, sb = _prep(mode, A, B, sa, sb)
    M, K = A.shape
    N = B.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    R = np.empty(ms.shape[0], dtype=np.float64)
    ref = np.empty(ms.shape[0], dtype=np.uint16)
    rc = lib().sgo_gemm_points(m, M, N, K, _ptr(A), _ptr(B), _ptr(sa), _ptr(sb), ms.shape[0], _ptr(ms), _ptr(ns), _ptr(R), _ptr(ref))
    if rc != 0:
        raise ValueError("oracle gemm_points rejected its arguments (rc=%d)" % rc)
    return R, ref


def gather_source(idx, rows_src):
    """For each output row of a gather-GEMM, the source row it reads and whether
    that row exists.  An index outside [0, rows_src) names no row: the output row
    reads row 0 with scale 0, so it is zero (this project's reading; ROCm/aiter
    PR 6539, Technical Details, names the gather_kv_b_proj kernel without fixing
    what a bad index does)."""
    idx = np.asarray(idx, dtype=np.int64)
    valid = (idx >= 0) & (idx < rows_src)
    return np.where(valid, idx, 0), valid


def gemm_gather(A_src, idx, B, sa_src, sb, rows=None, want_r=True):
    """Gather-GEMM in ptpc mode: output row i is the ptpc GEMM row of source row
    idx[i] of A_src [R, K] (e4m3) with its per-row scale sa_src[idx[i]], against B
    [N, K] with per-channel scales sb -- the gather of rows by index that
    gather_kv_b_proj fuses in front of the projection GEMM (ROCm/aiter PR 6539,
    Motivation and Technical Details).  The gather is numpy indexing; the GEMM is
    ``gemm("ptpc", ...)`` on the gathered rows.  Returns ``(R, ref)`` as gemm."""
    A_src = np.ascontiguousarray(A_src, dtype=np.uint8)
    sa_src = np.ascontiguousarray(sa_src, dtype=np.float32)
    src, valid = gather_source(idx, A_src.shape[0])
    A = A_src[src]
    sa = np.where(valid, sa_src[src], np.float32(0)).astype(np.float32)
    return gemm("ptpc", A, B, sa, sb, rows=rows, want_r=want_r)


def gemm_gather_points(A_src, idx, B, sa_src, sb, ms, ns):
    """Elements (ms[j], ns[j]) of the gather-GEMM, computed one by one."""
    A_src = np.ascontiguousarray(A_src, dtype=np.uint8)
    sa_src = np.ascontiguousarray(sa_src, dtype=np.float32)
    src, valid = gather_source(idx, A_src.shape[0])
    A = A_src[src]
    sa = np.where(valid, sa_src[src], np.float32(0)).astype(np.float32)
    return gemm_points("ptpc", A, B, sa, sb, ms, ns)


def bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values, via the oracle's own decoder rule."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_rne_sat(x) -> np.ndarray:
    """Nearest e4m3fn codes (ties to even, saturated to +-448) of binary64 values."""
    L = lib()
    v = np.asarray(x, dtype=np.float64)
    return np.array([L.sgo_e4m3_rne_sat(float(t)) for t in v.ravel()], dtype=np.uint8).reshape(v.shape)


def quantize(mode, X):
    """Quantise X [R, C] (float32, or uint16 bf16 bits) in `mode` ("ptpc",
    "blockscale" 1x128, "mxfp8" 1x32) into (codes uint8 [R, C], scales) with the
    scales in the GEMM's A-side layout: ptpc float32 [R]; blockscale float32
    [C/128, R]; mxfp8 uint8 e8m0 [C/32, R]."""
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    X = np.ascontiguousarray(X)
    bf16 = X.dtype == np.uint16
    if not bf16:
        X = X.astype(np.float32, copy=False)
    R, C = X.shape
    Q = np.empty((R, C), dtype=np.uint8)
    if m == 1:
        S = np.empty(R, dtype=np.float32)
    elif m == 2:
        S = np.empty((C // 128, R), dtype=np.float32)
    elif m == 3:
        S = np.empty((C // 32, R), dtype=np.uint8)
    else:
        raise ValueError("quantize: mode must be ptpc, blockscale or mxfp8")
    rc = lib().sgo_quantize(m, int(bf16), R, C, _ptr(X), _ptr(Q), _ptr(S))
    if rc != 0:
        raise ValueError("oracle quantize rejected its arguments (rc=%d)" % rc)
    return Q, S
