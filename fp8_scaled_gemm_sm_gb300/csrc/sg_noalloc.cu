// sg_noalloc.cu -- scaled_gemm_launch_noalloc: the ptpc GEMM for callers that
// cannot allocate device memory.
//
// The handle API (scaled_gemm_create) allocates the kernels' 16-byte watchdog
// status record with cudaMalloc.  Code that must not allocate -- for example
// inside a custom allocator or a memory-pool callback, where a nested
// cudaMalloc would re-enter the allocator, or in a process whose device memory
// is all reserved up front by a pool -- cannot use it.  This entry point launches the same ptpc kernel with
// that record in a file-scope static device array instead, so a launch performs
// no allocation at all: no cudaMalloc, no cudaFree, no allocating library call.
//
// The array is part of the library image: every GPU that loads the library holds
// it until the process exits.  Every call shares it and it keeps the previous
// call's contents, so each call clears it (cudaMemsetAsync on the caller's
// stream) before the kernel; calls whose kernels overlap on the GPU race on it.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "scaled_gemm.h"
#include "sg_internal.h"

namespace {

// Scratch of the no-allocation path: the kernel's watchdog status record
// (code, wait site, two spare words).  64 bytes is the stated maximum.
constexpr size_t kNoAllocScratchBytes = 64;
constexpr size_t kStatusRecordBytes = 16;
static_assert(kStatusRecordBytes <= kNoAllocScratchBytes, "status record must fit the static scratch");

static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

struct DeviceSetup {
  std::once_flag once;
  bool ok = false;
  int32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];

bool debug_on() {
  const char* e = std::getenv("SG_DEBUG");
  return e && *e && std::strcmp(e, "0") != 0;
}

sg_status_t reject(sg_status_t s, const char* what) {
  if (debug_on()) std::fprintf(stderr, "scaled_gemm_launch_noalloc: %s\n", what);
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device, with that device current: check it, look up the device
// address of the static scratch (the host-side symbol is only a stand-in), and
// set the kernel's shared-memory attribute.
void setup_device(int dev, DeviceSetup* s) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&s->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return;
  if (major != 10 || minor != 3) return;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return;
  if (sg::dense_prepare(sg::kModePtpcHost) != cudaSuccess) return;
  s->scratch = static_cast<int32_t*>(p);
  s->ok = true;
}

}  // namespace

extern "C" sg_status_t scaled_gemm_launch_noalloc(const void* A, const void* B, const void* a_scale,
                                                  const void* b_scale, void* C, int64_t M, int64_t N,
                                                  int64_t K, sg_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return reject(SG_ERR_INVALID_ARG, "negative size");
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return reject(SG_ERR_UNSUPPORTED_SHAPE, "size >= 2^31");
  if (N % 16 != 0) return reject(SG_ERR_UNSUPPORTED_SHAPE, "N % 16 != 0");
  if (K % 16 != 0) return reject(SG_ERR_UNSUPPORTED_SHAPE, "K % 16 != 0");
  if (K == 0) return reject(SG_ERR_UNSUPPORTED_SHAPE, "K == 0 (use scaled_gemm_launch)");
  if (M == 0 || N == 0) return SG_OK;
  if (!A || !B || !a_scale || !b_scale || !C) return reject(SG_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(a_scale) || !aligned16(b_scale) || !aligned16(C))
    return reject(SG_ERR_MISALIGNED, "pointer not 16-byte aligned");
  if (sg::ranges_overlap(C, M * N * 2, A, M * K) || sg::ranges_overlap(C, M * N * 2, B, N * K))
    return reject(SG_ERR_INVALID_ARG, "C overlaps A or B");
  if (sg::ranges_overlap(C, M * N * 2, a_scale, 4 * M) || sg::ranges_overlap(C, M * N * 2, b_scale, 4 * N))
    return reject(SG_ERR_INVALID_ARG, "C overlaps a scale buffer");
  // The only scratch this kernel needs is its status record.
  if (kStatusRecordBytes > kNoAllocScratchBytes)
    return reject(SG_ERR_UNSUPPORTED_SHAPE, "launch needs more scratch than the static array holds");

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return reject(SG_ERR_CUDA, "cudaGetDevice");
  if (dev >= kMaxDevices) return reject(SG_ERR_UNSUPPORTED_DEVICE, "device ordinal beyond the set-up table");
  DeviceSetup* s = &g_setup[dev];
  std::call_once(s->once, setup_device, dev, s);
  if (!s->ok) return reject(SG_ERR_UNSUPPORTED_DEVICE, "device set-up failed (not sm_103, or symbol lookup failed)");

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(s->scratch, 0, kStatusRecordBytes, st) != cudaSuccess)
    return reject(SG_ERR_CUDA, "clearing the status record");

  sg::LaunchArgs a{};
  a.mode = sg::kModePtpcHost;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = A;
  a.B = B;
  a.a_scale = a_scale;
  a.b_scale = b_scale;
  a.C = C;
  a.stream = st;
  a.num_sms = s->num_sms;
  a.status = s->scratch;
  a.timeout_ns = kTimeoutNs;
  a.skip_kstep = -1;
  const sg_status_t r = sg::dense_launch(a);
  return r == SG_OK ? SG_OK : reject(r, "kernel launch");
}
