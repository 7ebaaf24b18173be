// sg_internal.h -- host-side interface between the C ABI (scaled_gemm.cu) and
// the per-mode kernel launchers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "scaled_gemm.h"

namespace sg {

// Everything one launch needs, validated by the C ABI before any launcher runs.
struct LaunchArgs {
  int mode;
  int64_t M, N, K;
  const void* A;
  const void* B;
  const void* a_scale;
  const void* b_scale;
  void* C;
  cudaStream_t stream;
  int num_sms;
  int* status;          // device status word of the plan
  uint64_t timeout_ns;  // per-wait limit
  int32_t skip_kstep;   // watchdog tests: -1 = off
  void* workspace;      // the plan's device workspace (mxfp8: scale records), or NULL
  const int32_t* gather_idx;  // gather-GEMM: idx [M] (else NULL); A is then the source [rows_src][K]
  int64_t rows_src;
  int tile_bn;          // output-tile width pinned on the plan, or 0: chosen per launch
};

// Mode numbers as the launchers take them (equal to sg_mode_t).
constexpr int kModeBf16Host = SG_MODE_BF16;
constexpr int kModePtpcHost = SG_MODE_PTPC;

struct TileConfig {
  int bm, bn, bk, stages;
  int cluster;         // CTAs per cluster
  int rows_per_group;  // output rows one cluster covers per tile (N block) it takes
};

// Bytes of the A-side and B-side scale buffers of a launch (the layouts of
// include/scaled_gemm.h; 0 for bf16).
inline int64_t scale_bytes_a(int mode, int64_t M, int64_t K) {
  switch (mode) {
    case SG_MODE_PTPC: return 4 * M;
    case SG_MODE_BLOCKSCALE: return 4 * (K / 128) * M;
    case SG_MODE_MXFP8: return (K / 32) * M;
  }
  return 0;
}
inline int64_t scale_bytes_b(int mode, int64_t N, int64_t K) {
  switch (mode) {
    case SG_MODE_PTPC: return 4 * N;
    case SG_MODE_BLOCKSCALE: return 4 * ((N + 127) / 128) * (K / 128);
    case SG_MODE_MXFP8: return (K / 32) * N;
  }
  return 0;
}

// Whether the byte ranges [p, p + pb) and [q, q + qb) share a byte.
inline bool ranges_overlap(const void* p, int64_t pb, const void* q, int64_t qb) {
  if (!p || !q || pb <= 0 || qb <= 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + static_cast<uintptr_t>(qb) && b < a + static_cast<uintptr_t>(pb);
}

// Encode a 2D tiled TMA descriptor (inner dimension first).  Returns false if
// the driver rejects it.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle);

// Remember a CUDA error from a kernel launch for SG_DEBUG reporting (per thread).
void note_cuda_error(cudaError_t e);
const char* last_cuda_error();

// Launch configuration of the GEMM kernels: `cluster` CTAs per cluster (1: no
// cluster attribute) and programmatic stream serialization, so the launch may
// begin while the previous kernel in the stream finishes; the kernels wait in
// griddepcontrol.wait before touching global memory.  The attribute array lives
// in the object: construct it in place and pass `cfg`.
struct GemmLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2]{};
  GemmLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, unsigned cluster) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster > 1) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = cluster;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
  }
  GemmLaunch(const GemmLaunch&) = delete;
  GemmLaunch& operator=(const GemmLaunch&) = delete;
};

// cudaGetLastError after a launch, noted; SG_OK or SG_ERR_CUDA.
inline sg_status_t launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return SG_OK;
  note_cuda_error(e);
  return SG_ERR_CUDA;
}

int64_t quantize_max_cols();
sg_status_t quantize_launch(int mode, bool bf16, const void* X, int64_t R, int64_t C, void* Q,
                            void* scale, int num_sms, cudaStream_t st);

cudaError_t dense_prepare(int mode);
sg_status_t dense_launch(const LaunchArgs& a);
sg_status_t dense_launch_gather(const LaunchArgs& a);  // ptpc, A rows gathered by a.gather_idx
void dense_config(int mode, int64_t M, int64_t N, int num_sms, int tile_bn, TileConfig* c);
bool dense_tile_ok(int bn);  // a width scaled_gemm_set_tile may pin for ptpc / bf16

cudaError_t mxfp8_prepare();
size_t mxfp8_workspace_bytes(int64_t M_max, int64_t N, int64_t K);  // scale records
sg_status_t mxfp8_launch(const LaunchArgs& a);
void mxfp8_config(int64_t M, int64_t N, int num_sms, int tile_bn, TileConfig* c);
bool mxfp8_tile_ok(int bn);  // a width the mxfp8 kernels have

cudaError_t blockscale_prepare();
sg_status_t blockscale_launch(const LaunchArgs& a);
void blockscale_config(TileConfig* c);

}  // namespace sg
