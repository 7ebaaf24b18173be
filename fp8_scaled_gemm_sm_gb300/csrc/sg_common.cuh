// sg_common.cuh -- kernel parameters, tile scheduling and the epilogue shared by
// the sm_103a GEMM kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sg_ptx.cuh"

namespace sg {

enum Mode : int { kModeBf16 = 0, kModePtpc = 1, kModeBlockscale = 2, kModeMxfp8 = 3 };

constexpr int kBM = 128;          // output tile rows (one TMEM lane per row)
constexpr int kRowBytes = 128;    // bytes of K per operand row per pipeline stage
constexpr int kCBoxCols = 32;     // epilogue TMA store box: 32 bf16 columns ...
constexpr int kCBoxRows = 32;     // ... x 32 rows (one TMEM lane quarter)
constexpr int kCBoxBytes = kCBoxCols * kCBoxRows * 2;

struct GemmParams {
  int32_t M, N, K;
  int32_t m_blocks, n_blocks, k_blocks;
  int32_t num_tiles;
  int32_t skip_kstep;        // watchdog tests only: producer skips this stage (-1: never)
  const float* a_scale;      // ptpc [M]; blockscale [K/128][M]
  const float* b_scale;      // ptpc [N]; blockscale [ceil(N/128)][K/128]
  int* status;               // device status word
  uint64_t timeout_ns;       // limit of every mbarrier wait
};

// Persistent static schedule: CTA b takes tiles b, b + grid, b + 2*grid, ...
// Tiles are numbered with the N block fastest, so the CTAs in flight at any
// moment share a few A row panels and sweep all of B, which stays L2-resident.
struct TileCoord {
  int mb, nb;
};

__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int t) {
  TileCoord c;
  c.mb = t / p.n_blocks;
  c.nb = t - c.mb * p.n_blocks;
  return c;
}

// Address of the 16-byte chunk `chunk` (0..3) of row `row` in a 32 x 64-byte
// store box laid out with the TMA 64-byte swizzle (chunk bits 4-5 XOR address
// bits 7-8).  The box base is 512-byte aligned.
__device__ __forceinline__ uint32_t cbox_chunk_addr(uint32_t box, int row, int chunk) {
  return box + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Round 32 fp32 values of one row to bf16 and store the warp's 32 x 32 box.
// The warp owns two kCBoxBytes store boxes at `bufs` and alternates between them
// with the running counter `box`: the store that last read the box about to be
// written was committed two boxes ago, so at most one newer store may still be
// reading shared memory.  Every writer fences its generic stores into
// the async proxy before lane 0 issues the TMA store (deepseek-ai/DeepGEMM
// PR 453, Fix: the fence is executed by all threads, not only the issuing one).
__device__ __forceinline__ void store_box32(uint32_t bufs, uint32_t& box, const float (&f)[32],
                                            const CUtensorMap* tmC, int x, int y, int N, int M,
                                            int lane) {
  const uint32_t buf = bufs + (box & 1u) * kCBoxBytes;
  ++box;
  uint32_t packed[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(f[2 * j], f[2 * j + 1]);
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_shared_v4(cbox_chunk_addr(buf, lane, k), packed[4 * k], packed[4 * k + 1], packed[4 * k + 2],
                 packed[4 * k + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (x < N && y < M) tma_store_2d(tmC, buf, x, y);
    bulk_commit_group();
  }
}

// Epilogue worker for one output tile, run by one warp on 32 rows (its TMEM lane
// quarter) and NCOLS columns starting at the accumulator address `taddr`.  Values
// are read from TMEM, multiplied by `row_scale * col_scale[c]` when SCALED,
// rounded to bf16 and stored through the warp's two store boxes `bufs` (box
// counter `box`).  `release()` runs once, right after the last TMEM load.
template <int NCOLS, bool SCALED, typename Release>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, uint32_t bufs, uint32_t& box,
                                              const float* col_scale,
                                              float row_scale, const CUtensorMap* tmC, int n_start,
                                              int m_start, int N, int M, int lane,
                                              Release&& release) {
  static_assert(NCOLS % 32 == 0, "epilogue works in 32-column boxes");
  auto convert = [&](const uint32_t (&v)[32], int cc, float (&f)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      f[j] = __uint_as_float(v[j]);
      if constexpr (SCALED) f[j] = f[j] * row_scale * col_scale[cc + j];
    }
  };
#pragma unroll 1
  for (int c = 0; c + 64 <= NCOLS; c += 64) {
    uint32_t v0[32], v1[32];
    tmem_ld_32x32b_x32(taddr + c, v0);
    tmem_ld_32x32b_x32(taddr + c + 32, v1);
    tmem_wait_ld();
    if (c + 64 == NCOLS) release();
    float f[32];
    convert(v0, c, f);
    store_box32(bufs, box, f, tmC, n_start + c, m_start, N, M, lane);
    convert(v1, c + 32, f);
    store_box32(bufs, box, f, tmC, n_start + c + 32, m_start, N, M, lane);
  }
  if constexpr (NCOLS % 64 == 32) {
    constexpr int c = NCOLS - 32;
    uint32_t v0[32];
    tmem_ld_32x32b_x32(taddr + c, v0);
    tmem_wait_ld();
    release();
    float f[32];
    convert(v0, c, f);
    store_box32(bufs, box, f, tmC, n_start + c, m_start, N, M, lane);
  }
}

}  // namespace sg
