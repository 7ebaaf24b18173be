// scaled_gemm.cu -- the C ABI of libscaledgemm.so: plan creation, argument
// validation, TMA descriptor encoding and dispatch to the per-mode launchers.
// The shape and operand rules follow ROCm/mori PR 809 ("Using it": one plan per
// (n, k) serving any M up to m_max; operands the launch would misread are
// refused; N any multiple of 16) and are listed in include/scaled_gemm.h.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cuda.h>
#include <cuda_runtime.h>

#include "scaled_gemm.h"
#include "sg_internal.h"

struct sg_gemm {
  int mode;
  int64_t N, K, M_max;
  int device;
  int num_sms;
  int* status;  // device: [code, where, 0, 0]
  void* workspace;  // device; mxfp8: the scale records of one launch (else NULL)
  uint64_t timeout_ns;
  int32_t skip_kstep;
  int tile_bn;  // output-tile width pinned by scaled_gemm_set_tile, or 0
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;

bool debug_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("SG_DEBUG");
    return e && *e && std::strcmp(e, "0") != 0;
  }();
  return on;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

sg_status_t fail(sg_status_t s, const char* what) {
  if (debug_enabled()) {
    if (s == SG_ERR_CUDA && g_last_cuda_error != cudaSuccess)
      std::fprintf(stderr, "scaled_gemm: %s (%s: %s)\n", what, scaled_gemm_status_string(s),
                   cudaGetErrorString(g_last_cuda_error));
    else
      std::fprintf(stderr, "scaled_gemm: %s (%s)\n", what, scaled_gemm_status_string(s));
  }
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// K granularity per mode.
int64_t k_multiple(int mode) {
  switch (mode) {
    case SG_MODE_PTPC: return 16;
    case SG_MODE_BF16: return 8;
    case SG_MODE_BLOCKSCALE: return 128;
    case SG_MODE_MXFP8: return 32;
  }
  return 0;
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

}  // namespace

namespace sg {

void note_cuda_error(cudaError_t e) { g_last_cuda_error = e; }
const char* last_cuda_error() { return cudaGetErrorString(g_last_cuda_error); }

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sg

extern "C" {

const char* scaled_gemm_status_string(sg_status_t s) {
  switch (s) {
    case SG_OK: return "ok";
    case SG_ERR_INVALID_ARG: return "invalid argument";
    case SG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SG_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SG_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    case SG_ERR_CUDA: return "CUDA error";
    case SG_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

sg_status_t scaled_gemm_create(sg_handle_t* out, int mode, int64_t N, int64_t K, int64_t M_max,
                               int device) {
  if (!out) return fail(SG_ERR_INVALID_ARG, "create: out is NULL");
  *out = nullptr;
  if (mode < SG_MODE_BF16 || mode > SG_MODE_MXFP8) return fail(SG_ERR_INVALID_ARG, "create: bad mode");
  if (N < 0 || K < 0 || M_max < 0) return fail(SG_ERR_INVALID_ARG, "create: negative size");
  if (N > kMaxDim || K > kMaxDim || M_max > kMaxDim) return fail(SG_ERR_UNSUPPORTED_SHAPE, "create: size >= 2^31");
  if (N % 16 != 0) return fail(SG_ERR_UNSUPPORTED_SHAPE, "create: N % 16 != 0");
  if (K % k_multiple(mode) != 0) return fail(SG_ERR_UNSUPPORTED_SHAPE, "create: K not a multiple of the mode's block");
  if (N > 0 && K > 0 && (N * K) / K != N) return fail(SG_ERR_UNSUPPORTED_SHAPE, "create: N*K overflows");

  int dev = device;
  if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) return fail(SG_ERR_CUDA, "create: cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(SG_ERR_CUDA, "create: device query");
  if (major != 10 || minor != 3) return fail(SG_ERR_UNSUPPORTED_DEVICE, "create: not compute capability 10.3");
  if (!encode_tiled_fn()) return fail(SG_ERR_CUDA, "create: cuTensorMapEncodeTiled unavailable");

  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return fail(SG_ERR_CUDA, "create: cudaSetDevice");
  cudaError_t e = cudaSuccess;
  switch (mode) {
    case SG_MODE_BF16:
    case SG_MODE_PTPC: e = sg::dense_prepare(mode); break;
    case SG_MODE_MXFP8: e = sg::mxfp8_prepare(); break;
    case SG_MODE_BLOCKSCALE: e = sg::blockscale_prepare(); break;
  }
  int* status = nullptr;
  void* workspace = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&status, 16);
  if (e == cudaSuccess) e = cudaMemset(status, 0, 16);
  const size_t ws_bytes = mode == SG_MODE_MXFP8 ? sg::mxfp8_workspace_bytes(M_max, N, K) : 0;
  if (e == cudaSuccess && ws_bytes > 0) e = cudaMalloc(&workspace, ws_bytes);
  if (prev >= 0 && prev != dev) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    if (status) cudaFree(status);
    if (workspace) cudaFree(workspace);
    return fail(SG_ERR_CUDA, "create: kernel attributes / status word / workspace");
  }
  sg_gemm* h = new (std::nothrow) sg_gemm;
  if (!h) {
    cudaFree(status);
    if (workspace) cudaFree(workspace);
    return fail(SG_ERR_CUDA, "create: out of host memory");
  }
  h->mode = mode;
  h->N = N;
  h->K = K;
  h->M_max = M_max;
  h->device = dev;
  h->num_sms = sms;
  h->status = status;
  h->workspace = workspace;
  h->timeout_ns = kDefaultTimeoutNs;
  h->skip_kstep = -1;
  h->tile_bn = 0;
  *out = h;
  return SG_OK;
}

sg_status_t scaled_gemm_destroy(sg_handle_t h) {
  if (!h) return SG_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != h->device) cudaSetDevice(h->device);
  cudaError_t e = cudaFree(h->status);
  if (h->workspace) {
    const cudaError_t e2 = cudaFree(h->workspace);
    if (e == cudaSuccess) e = e2;
  }
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  delete h;
  return e == cudaSuccess ? SG_OK : SG_ERR_CUDA;
}

sg_status_t scaled_gemm_get_config(sg_handle_t h, int* bm, int* bn, int* bk, int* stages, int* grid) {
  if (!h) return fail(SG_ERR_INVALID_ARG, "get_config: NULL handle");
  sg::TileConfig c{};
  switch (h->mode) {
    case SG_MODE_BF16:
    case SG_MODE_PTPC: sg::dense_config(h->mode, h->M_max, h->N, h->num_sms, h->tile_bn, &c); break;
    case SG_MODE_MXFP8: sg::mxfp8_config(h->M_max, h->N, h->num_sms, h->tile_bn, &c); break;
    case SG_MODE_BLOCKSCALE: sg::blockscale_config(&c); break;
  }
  if (bm) *bm = c.bm;
  if (bn) *bn = c.bn;
  if (bk) *bk = c.bk;
  if (stages) *stages = c.stages;
  if (grid) {  // the launch's persistent CTAs: whole clusters, at most one CTA per SM
    const int64_t groups = ((h->M_max + c.rows_per_group - 1) / c.rows_per_group) * ((h->N + c.bn - 1) / c.bn);
    const int64_t max_groups = h->num_sms / c.cluster;
    *grid = static_cast<int>((groups < max_groups ? groups : max_groups) * c.cluster);
  }
  return SG_OK;
}

sg_status_t scaled_gemm_set_tile(sg_handle_t h, int bn) {
  if (!h) return fail(SG_ERR_INVALID_ARG, "set_tile: NULL handle");
  if (bn == 0) {
    h->tile_bn = 0;
    return SG_OK;
  }
  sg::TileConfig c{};
  bool ok = false;
  switch (h->mode) {
    case SG_MODE_MXFP8: ok = sg::mxfp8_tile_ok(bn); break;
    case SG_MODE_BF16:
    case SG_MODE_PTPC: ok = sg::dense_tile_ok(bn); break;
    case SG_MODE_BLOCKSCALE: sg::blockscale_config(&c); ok = bn == c.bn; break;
  }
  if (!ok) return fail(SG_ERR_INVALID_ARG, "set_tile: a width this mode does not have");
  h->tile_bn = bn;
  return SG_OK;
}

sg_status_t scaled_gemm_set_debug(sg_handle_t h, int64_t timeout_ns, int64_t skip_kstep) {
  if (!h) return fail(SG_ERR_INVALID_ARG, "set_debug: NULL handle");
  if (timeout_ns < 0 || skip_kstep < -1 || skip_kstep > kMaxDim) return fail(SG_ERR_INVALID_ARG, "set_debug: bad value");
  h->timeout_ns = timeout_ns ? static_cast<uint64_t>(timeout_ns) : kDefaultTimeoutNs;
  h->skip_kstep = static_cast<int32_t>(skip_kstep);
  return SG_OK;
}

sg_status_t scaled_gemm_debug_status(sg_handle_t h, sg_stream_t stream, int32_t* code, int32_t* where) {
  if (!h || !code) return fail(SG_ERR_INVALID_ARG, "debug_status: NULL argument");
  int32_t host[4] = {0, 0, 0, 0};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host, h->status, 16, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(h->status, 0, 16, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return fail(SG_ERR_CUDA, "debug_status: copy");
  *code = host[0];
  if (where) *where = host[0] ? host[1] : 0;
  return SG_OK;
}

sg_status_t scaled_gemm_launch(sg_handle_t h, const void* A, const void* B, const void* a_scale,
                               const void* b_scale, void* C, int64_t M, sg_stream_t stream) {
  if (!h) return fail(SG_ERR_INVALID_ARG, "launch: NULL handle");
  if (M < 0 || M > h->M_max) return fail(SG_ERR_INVALID_ARG, "launch: M outside [0, M_max]");
  if (M == 0 || h->N == 0) return SG_OK;
  const bool scaled = h->mode != SG_MODE_BF16;
  if (!C) return fail(SG_ERR_INVALID_ARG, "launch: C is NULL");
  if (!aligned16(C)) return fail(SG_ERR_MISALIGNED, "launch: C");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (h->K == 0) {  // empty contraction: C = 0
    return cudaMemsetAsync(C, 0, static_cast<size_t>(M) * h->N * 2, s) == cudaSuccess
               ? SG_OK
               : fail(SG_ERR_CUDA, "launch: memset");
  }
  if (!A || !B) return fail(SG_ERR_INVALID_ARG, "launch: A or B is NULL");
  if (scaled && (!a_scale || !b_scale)) return fail(SG_ERR_INVALID_ARG, "launch: scales are NULL");
  if (!scaled && (a_scale || b_scale)) return fail(SG_ERR_INVALID_ARG, "launch: bf16 takes no scales");
  if (!aligned16(A) || !aligned16(B)) return fail(SG_ERR_MISALIGNED, "launch: A or B");
  if (scaled && (!aligned16(a_scale) || !aligned16(b_scale))) return fail(SG_ERR_MISALIGNED, "launch: scales");
  // C must not overlap an operand or a scale buffer (the kernel streams C out
  // while it still reads them).
  const int64_t el = h->mode == SG_MODE_BF16 ? 2 : 1;
  const int64_t cb = M * h->N * 2;
  if (sg::ranges_overlap(C, cb, A, M * h->K * el) || sg::ranges_overlap(C, cb, B, h->N * h->K * el))
    return fail(SG_ERR_INVALID_ARG, "launch: C overlaps A or B");
  if (sg::ranges_overlap(C, cb, a_scale, sg::scale_bytes_a(h->mode, M, h->K)) ||
      sg::ranges_overlap(C, cb, b_scale, sg::scale_bytes_b(h->mode, h->N, h->K)))
    return fail(SG_ERR_INVALID_ARG, "launch: C overlaps a scale buffer");

  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return fail(SG_ERR_CUDA, "launch: cudaGetDevice");
  if (cur != h->device) return fail(SG_ERR_INVALID_ARG, "launch: current device differs from the plan's");

  sg::LaunchArgs a{};
  a.mode = h->mode;
  a.M = M;
  a.N = h->N;
  a.K = h->K;
  a.A = A;
  a.B = B;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.C = C;
  a.stream = s;
  a.num_sms = h->num_sms;
  a.status = h->status;
  a.timeout_ns = h->timeout_ns;
  a.skip_kstep = h->skip_kstep;
  a.tile_bn = h->tile_bn;
  a.workspace = h->workspace;
  sg_status_t r = SG_ERR_INVALID_ARG;
  switch (h->mode) {
    case SG_MODE_BF16:
    case SG_MODE_PTPC: r = sg::dense_launch(a); break;
    case SG_MODE_MXFP8: r = sg::mxfp8_launch(a); break;
    case SG_MODE_BLOCKSCALE: r = sg::blockscale_launch(a); break;
  }
  return r == SG_OK ? SG_OK : fail(r, "launch: kernel launch");
}

sg_status_t scaled_gemm_launch_gather(sg_handle_t h, const void* A_src, int64_t R, const int32_t* idx,
                                      const void* B, const void* a_scale_src, const void* b_scale,
                                      void* C, int64_t M, sg_stream_t stream) {
  if (!h) return fail(SG_ERR_INVALID_ARG, "launch_gather: NULL handle");
  if (h->mode != SG_MODE_PTPC) return fail(SG_ERR_INVALID_ARG, "launch_gather: the plan is not ptpc");
  if (M < 0 || M > h->M_max) return fail(SG_ERR_INVALID_ARG, "launch_gather: M outside [0, M_max]");
  if (R < 0) return fail(SG_ERR_INVALID_ARG, "launch_gather: negative R");
  if (R > kMaxDim) return fail(SG_ERR_UNSUPPORTED_SHAPE, "launch_gather: R >= 2^31");
  if (M == 0 || h->N == 0) return SG_OK;
  if (!C) return fail(SG_ERR_INVALID_ARG, "launch_gather: C is NULL");
  if (!aligned16(C)) return fail(SG_ERR_MISALIGNED, "launch_gather: C");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (h->K == 0 || R == 0) {  // empty contraction, or no source row: C = 0
    return cudaMemsetAsync(C, 0, static_cast<size_t>(M) * h->N * 2, s) == cudaSuccess
               ? SG_OK
               : fail(SG_ERR_CUDA, "launch_gather: memset");
  }
  if (!A_src || !idx || !B || !a_scale_src || !b_scale)
    return fail(SG_ERR_INVALID_ARG, "launch_gather: NULL operand");
  if (!aligned16(A_src) || !aligned16(idx) || !aligned16(B) || !aligned16(a_scale_src) || !aligned16(b_scale))
    return fail(SG_ERR_MISALIGNED, "launch_gather: operand");
  const int64_t cb = M * h->N * 2;
  if (sg::ranges_overlap(C, cb, A_src, R * h->K) || sg::ranges_overlap(C, cb, B, h->N * h->K) ||
      sg::ranges_overlap(C, cb, idx, M * 4) || sg::ranges_overlap(C, cb, a_scale_src, 4 * R) ||
      sg::ranges_overlap(C, cb, b_scale, 4 * h->N))
    return fail(SG_ERR_INVALID_ARG, "launch_gather: C overlaps an operand or a scale buffer");
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return fail(SG_ERR_CUDA, "launch_gather: cudaGetDevice");
  if (cur != h->device) return fail(SG_ERR_INVALID_ARG, "launch_gather: current device differs from the plan's");

  sg::LaunchArgs a{};
  a.mode = h->mode;
  a.M = M;
  a.N = h->N;
  a.K = h->K;
  a.A = A_src;
  a.B = B;
  a.a_scale = a_scale_src;
  a.b_scale = b_scale;
  a.C = C;
  a.stream = s;
  a.num_sms = h->num_sms;
  a.status = h->status;
  a.timeout_ns = h->timeout_ns;
  a.skip_kstep = h->skip_kstep;
  a.tile_bn = h->tile_bn;
  a.gather_idx = idx;
  a.rows_src = R;
  const sg_status_t r = sg::dense_launch_gather(a);
  return r == SG_OK ? SG_OK : fail(r, "launch_gather: kernel launch");
}

sg_status_t scaled_gemm_quantize(int mode, int x_dtype, const void* X, int64_t R, int64_t C, void* Q,
                                 void* scale, sg_stream_t stream) {
  if (mode != SG_MODE_PTPC && mode != SG_MODE_BLOCKSCALE && mode != SG_MODE_MXFP8)
    return fail(SG_ERR_INVALID_ARG, "quantize: mode must be ptpc, blockscale or mxfp8");
  if (x_dtype != SG_DTYPE_BF16 && x_dtype != SG_DTYPE_F32) return fail(SG_ERR_INVALID_ARG, "quantize: bad x_dtype");
  if (R < 0 || C < 0) return fail(SG_ERR_INVALID_ARG, "quantize: negative size");
  if (R > kMaxDim || C > sg::quantize_max_cols()) return fail(SG_ERR_UNSUPPORTED_SHAPE, "quantize: R >= 2^31 or C > 32768");
  if (C % k_multiple(mode) != 0) return fail(SG_ERR_UNSUPPORTED_SHAPE, "quantize: C not a multiple of the mode's block");
  if (R == 0 || C == 0) return SG_OK;
  if (!X || !Q || !scale) return fail(SG_ERR_INVALID_ARG, "quantize: NULL pointer");
  if (!aligned16(X) || !aligned16(Q) || !aligned16(scale)) return fail(SG_ERR_MISALIGNED, "quantize: pointer");
  int dev = -1, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(SG_ERR_CUDA, "quantize: device query");
  const sg_status_t r = sg::quantize_launch(mode, x_dtype == SG_DTYPE_BF16, X, R, C, Q, scale, sms,
                                            reinterpret_cast<cudaStream_t>(stream));
  return r == SG_OK ? SG_OK : fail(r, "quantize: kernel launch");
}

}  // extern "C"
