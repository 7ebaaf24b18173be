"""GB300 (sm_103a) scaled FP8 / BF16 GEMM.

``C[M,N] = bf16((A[M,K] . B[N,K]^T) scaled)`` with fp32 accumulation, in the
ptpc, blockscale, mxfp8 and bf16 modes, computed by hand-written tcgen05 / TMA
kernels in ``libscaledgemm.so`` (C ABI: ``include/scaled_gemm.h``).

``binding`` is a thin ctypes layer with the C ABI's names; ``ScaledGemm`` wraps
it for torch CUDA tensors.  There is no fallback: if the library is missing or
the device is not sm_103, calls raise.  Importing the package loads nothing;
the library is loaded by the first call.
"""
from .binding import MODES, ScaledGemm, ScaledGemmError  # noqa: F401
