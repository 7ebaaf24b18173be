"""ctypes binding of libscaledgemm.so, with the C ABI's own names.

Argument marshalling only: every step of the GEMM runs in the library's CUDA
kernels.  Pointers are plain integers (device addresses), streams are raw
``cudaStream_t`` values (0 = legacy default stream).  A non-OK status raises
``ScaledGemmError``.  The library is never replaced by another implementation:
if it cannot be loaded, ``lib()`` raises.
"""
import ctypes
import os

MODES = {"bf16": 0, "ptpc": 1, "blockscale": 2, "mxfp8": 3}
STATUS = {
    0: "SG_OK",
    1: "SG_ERR_INVALID_ARG",
    2: "SG_ERR_UNSUPPORTED_SHAPE",
    3: "SG_ERR_MISALIGNED",
    4: "SG_ERR_UNSUPPORTED_DEVICE",
    5: "SG_ERR_CUDA",
    6: "SG_ERR_TIMEOUT",
}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libscaledgemm.so")

# Exported symbols and their signatures (the declarations of include/scaled_gemm.h).
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_int = ctypes.c_int
SIGNATURES = {
    "scaled_gemm_create": (_int, [ctypes.POINTER(_vp), _int, _i64, _i64, _i64, _int]),
    "scaled_gemm_launch": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "scaled_gemm_launch_gather": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _i64, _vp]),
    "scaled_gemm_destroy": (_int, [_vp]),
    "scaled_gemm_status_string": (ctypes.c_char_p, [_int]),
    "scaled_gemm_get_config": (_int, [_vp] + [ctypes.POINTER(_int)] * 5),
    "scaled_gemm_set_tile": (_int, [_vp, _int]),
    "scaled_gemm_debug_status": (_int, [_vp, _vp, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "scaled_gemm_set_debug": (_int, [_vp, _i64, _i64]),
    "scaled_gemm_launch_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "scaled_gemm_quantize": (_int, [_int, _int, _vp, _i64, _i64, _vp, _vp, _vp]),
}
DTYPES = {"bf16": 0, "f32": 1}


class ScaledGemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        name = STATUS.get(self.status, "status %d" % self.status)
        super().__init__("%s: %s%s" % (what, name, "" if not _LIB else " (%s)" % scaled_gemm_status_string(status)))


_LIB = None


def lib():
    """Load libscaledgemm.so (built by ``fp8_scaled_gemm_sm_gb300.build``)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libscaledgemm.so is not built; run `python -c 'import __graft_entry__ as g; g.build()'`"
            )
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status, what):
    if status != 0:
        raise ScaledGemmError(status, what)


def scaled_gemm_status_string(status):
    return lib().scaled_gemm_status_string(int(status)).decode()


def scaled_gemm_create(mode, N, K, M_max, device=-1):
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    h = _vp()
    _check(lib().scaled_gemm_create(ctypes.byref(h), m, int(N), int(K), int(M_max), int(device)), "scaled_gemm_create")
    return h.value


def scaled_gemm_launch(h, A, B, a_scale, b_scale, C, M, stream=0):
    _check(
        lib().scaled_gemm_launch(h, A, B, a_scale or None, b_scale or None, C, int(M), stream or None),
        "scaled_gemm_launch",
    )


def scaled_gemm_launch_gather(h, A_src, R, idx, B, a_scale_src, b_scale, C, M, stream=0):
    """Gather-GEMM on a ptpc plan: row i of C from source row idx[i] of A_src (see the C header)."""
    _check(
        lib().scaled_gemm_launch_gather(h, A_src or None, int(R), idx or None, B or None, a_scale_src or None,
                                        b_scale or None, C or None, int(M), stream or None),
        "scaled_gemm_launch_gather",
    )


def scaled_gemm_launch_noalloc(A, B, a_scale, b_scale, C, M, N, K, stream=0):
    """ptpc launch without a handle and without any device allocation (see the C header)."""
    _check(
        lib().scaled_gemm_launch_noalloc(A, B, a_scale, b_scale, C, int(M), int(N), int(K), stream or None),
        "scaled_gemm_launch_noalloc",
    )


def scaled_gemm_quantize(mode, x_dtype, X, R, C, Q, scale, stream=0):
    """Quantise X [R, C] (device pointer) to e4m3 codes Q and scales (see the C header)."""
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    dt = DTYPES[x_dtype] if isinstance(x_dtype, str) else int(x_dtype)
    _check(lib().scaled_gemm_quantize(m, dt, X, int(R), int(C), Q, scale, stream or None), "scaled_gemm_quantize")


def quantize(mode, x, stream=None):
    """Quantise a CUDA tensor x [R, C] (bfloat16 or float32) for `mode`; returns
    (codes uint8 [R, C], scales) with scales float32 [R] (ptpc), float32
    [C/128, R] (blockscale) or uint8 [C/32, R] (mxfp8)."""
    import torch

    if x.dtype not in (torch.bfloat16, torch.float32) or x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("quantize: x must be a contiguous 2-D bfloat16 or float32 CUDA tensor")
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    if mode == "ptpc":
        s = torch.empty(R, dtype=torch.float32, device=x.device)
    elif mode == "blockscale":
        s = torch.empty((C // 128, R), dtype=torch.float32, device=x.device)
    elif mode == "mxfp8":
        s = torch.empty((C // 32, R), dtype=torch.uint8, device=x.device)
    else:
        raise ValueError("quantize: mode must be ptpc, blockscale or mxfp8")
    st = torch.cuda.current_stream(x.device).cuda_stream if stream is None else stream
    scaled_gemm_quantize(mode, "bf16" if x.dtype == torch.bfloat16 else "f32", x.data_ptr(), R, C,
                         q.data_ptr(), s.data_ptr(), st)
    return q, s


def scaled_gemm_destroy(h):
    _check(lib().scaled_gemm_destroy(h), "scaled_gemm_destroy")


def scaled_gemm_get_config(h):
    v = [_int() for _ in range(5)]
    _check(lib().scaled_gemm_get_config(h, *[ctypes.byref(x) for x in v]), "scaled_gemm_get_config")
    return dict(zip(("bm", "bn", "bk", "stages", "grid"), (x.value for x in v)))


def scaled_gemm_debug_status(h, stream=0):
    code, where = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().scaled_gemm_debug_status(h, stream or None, ctypes.byref(code), ctypes.byref(where)), "scaled_gemm_debug_status")
    return code.value, where.value


def scaled_gemm_set_tile(h, bn=0):
    _check(lib().scaled_gemm_set_tile(h, int(bn)), "scaled_gemm_set_tile")


def scaled_gemm_set_debug(h, timeout_ns=0, skip_kstep=-1):
    _check(lib().scaled_gemm_set_debug(h, int(timeout_ns), int(skip_kstep)), "scaled_gemm_set_debug")


class ScaledGemm:
    """A plan for one (mode, N, K) serving any M <= M_max, for torch CUDA tensors.

    ``gemm(A, B, a_scale, b_scale, out=None)`` launches on torch's current
    stream and returns C [M, N] bf16.  A and B are uint8 (e4m3 codes) or
    float8_e4m3fn tensors in the fp8 modes and bfloat16 tensors in bf16 mode;
    scale layouts are those of include/scaled_gemm.h.
    """

    def __init__(self, mode, N, K, M_max, device=None):
        import torch

        self.mode = mode
        self.N, self.K, self.M_max = int(N), int(K), int(M_max)
        dev = torch.cuda.current_device() if device is None else int(device)
        self.device = dev
        self.handle = scaled_gemm_create(mode, N, K, M_max, dev)

    def config(self):
        return scaled_gemm_get_config(self.handle)

    def set_tile(self, bn=0):
        """Pin the output-tile width of later calls (mxfp8: 224 or 128; ptpc and
        bf16: 256 or 128; blockscale: 256), or 0 to let each call choose from its M."""
        scaled_gemm_set_tile(self.handle, bn)

    def __call__(self, A, B, a_scale=None, b_scale=None, out=None, stream=None):
        import torch

        M = A.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.bfloat16, device=A.device)
        for t in (A, B, out, a_scale, b_scale):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("operands must be contiguous CUDA tensors")
        if tuple(A.shape) != (M, self.K) or tuple(B.shape) != (self.N, self.K) or tuple(out.shape) != (M, self.N):
            raise ValueError("shape mismatch: A %s, B %s, out %s for N=%d K=%d" % (tuple(A.shape), tuple(B.shape), tuple(out.shape), self.N, self.K))
        s = torch.cuda.current_stream(A.device).cuda_stream if stream is None else stream
        scaled_gemm_launch(
            self.handle, A.data_ptr(), B.data_ptr(),
            a_scale.data_ptr() if a_scale is not None else 0,
            b_scale.data_ptr() if b_scale is not None else 0,
            out.data_ptr(), M, s,
        )
        return out

    def close(self):
        if getattr(self, "handle", None):
            scaled_gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
