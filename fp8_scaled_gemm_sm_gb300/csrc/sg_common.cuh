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

// Epilogue worker for one output tile, run by one warp on 32 rows (its TMEM lane
// quarter) and columns [col0, col0 + ncols) of the tile.  Values are read from
// TMEM, multiplied by `row_scale * col_scale[c]` when the mode has scales, rounded
// to bf16 and stored through two alternating 2 KB shared-memory boxes by TMA.
//
//   taddr      TMEM address of (lane quarter base, accumulator column col0)
//   bufs       two kCBoxBytes store boxes owned by this warp
//   col_scale  per-column scales in shared memory (nullptr: no scaling)
//   release    called once after the last TMEM load has completed
template <int NCOLS, bool SCALED, typename Release>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, uint32_t bufs, const float* col_scale,
                                              float row_scale, const CUtensorMap* tmC, int n_start,
                                              int m_start, int N, int M, int lane,
                                              Release&& release) {
  static_assert(NCOLS % 64 == 0, "epilogue works in 64-column steps");
#pragma unroll 1
  for (int c = 0; c < NCOLS; c += 64) {
    uint32_t v0[32], v1[32];
    tmem_ld_32x32b_x32(taddr + c, v0);
    tmem_ld_32x32b_x32(taddr + c + 32, v1);
    tmem_wait_ld();
    if (c + 64 == NCOLS) release();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t* v = half ? v1 : v0;
      const int cc = c + half * 32;
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float f0 = __uint_as_float(v[2 * j]);
        float f1 = __uint_as_float(v[2 * j + 1]);
        if constexpr (SCALED) {
          f0 = f0 * row_scale * col_scale[cc + 2 * j];
          f1 = f1 * row_scale * col_scale[cc + 2 * j + 1];
        }
        packed[j] = pack_bf16x2(f0, f1);
      }
      const uint32_t buf = bufs + half * kCBoxBytes;
      // The store that last read this box was committed two boxes ago.
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_shared_v4(cbox_chunk_addr(buf, lane, k), packed[4 * k], packed[4 * k + 1],
                     packed[4 * k + 2], packed[4 * k + 3]);
      // Every writer orders its generic stores before the async-proxy read.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (n_start + cc < N && m_start < M) tma_store_2d(tmC, buf, n_start + cc, m_start);
        bulk_commit_group();
      }
    }
  }
}

}  // namespace sg
