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
constexpr int kCBoxCols = 32;     // default epilogue TMA store box: 32 bf16 columns ...
constexpr int kCBoxRows = 32;     // ... x 32 rows (one TMEM lane quarter)
constexpr int kCBoxBytes = kCBoxCols * kCBoxRows * 2;

// Bytes of one warp's store box of W bf16 columns x 32 rows.
template <int W>
__host__ __device__ constexpr int cbox_bytes() {
  return W * kCBoxRows * 2;
}

struct GemmParams {
  int32_t M, N, K;
  int32_t m_blocks, n_blocks, k_blocks;
  int32_t num_tiles;
  int32_t skip_kstep;        // watchdog tests only: producer skips this stage (-1: never)
  const float* a_scale;      // ptpc [M]; blockscale [K/128][M]
  const float* b_scale;      // ptpc [N]; blockscale [ceil(N/128)][K/128]
  int* status;               // device status word
  uint64_t timeout_ns;       // limit of every mbarrier wait
  const void* a_src;         // gather-GEMM: the source A [rows_src][K] e4m3 (else NULL)
  const int32_t* gather_idx; // gather-GEMM: source row of each output row [M] (else NULL)
  int32_t rows_src;          // gather-GEMM: rows of the source A (and of a_scale)
};

// Persistent static schedule: CTA pair (or CTA group) g takes tiles g, g + G,
// g + 2G, ...  Tiles are numbered with the N block fastest, so the groups in
// flight at any moment share a few A row panels and sweep all of B, which stays
// L2-resident.  Each kernel maps a tile number to the 128-row block of its CTA.
struct TileCoord {
  int mb, nb;  // 128-row block of M, BN-column block of N
};

// Address of the 16-byte chunk `chunk` of row `row` in a 32-row store box of W
// bf16 columns, laid out with the TMA swizzle of its row width: W = 32 (64-byte
// rows, 64-byte swizzle: chunk bits 4-5 XOR address bits 7-8) or W = 64
// (128-byte rows, 128-byte swizzle: chunk bits 4-6 XOR address bits 7-9).
// The box base is 1024-byte aligned.
template <int W = 32>
__device__ __forceinline__ uint32_t cbox_chunk_addr(uint32_t box, int row, int chunk) {
  if constexpr (W == 32)
    return box + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
  else
    return box + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Round 32 fp32 values of one row to bf16 and store the warp's 32 x 32 box.
// The warp owns NBOX kCBoxBytes store boxes at `bufs` and cycles through them
// with the running counter `box`: the store that last read the box about to be
// written was committed NBOX boxes ago, so at most NBOX - 1 newer stores may
// still be reading shared memory.  Every writer fences its generic stores into
// the async proxy before lane 0 issues the TMA store (deepseek-ai/DeepGEMM
// PR 453, Fix: the fence is executed by all threads, not only the issuing one).
// The output is stored with the evict-first L2 policy: it is not read again.
template <int NBOX = 2, int W = 32>
__device__ __forceinline__ void store_box(uint32_t bufs, uint32_t& box, const uint32_t (&packed)[W / 2],
                                          const CUtensorMap* tmC, int x, int y, int N, int M, int lane) {
  static_assert(NBOX == 1 || NBOX == 2 || NBOX == 4, "boxes per warp");
  static_assert(W == 32 || W == 64, "box width");
  const uint32_t buf = bufs + (box & (NBOX - 1)) * cbox_bytes<W>();
  ++box;
  if (lane == 0) bulk_wait_group_read<NBOX - 1>();
  __syncwarp();
#pragma unroll
  for (int k = 0; k < W / 8; ++k)
    st_shared_v4(cbox_chunk_addr<W>(buf, lane, k), packed[4 * k], packed[4 * k + 1], packed[4 * k + 2],
                 packed[4 * k + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (x < N && y < M) tma_store_2d_hint(tmC, buf, x, y, l2_policy_evict_first());
    bulk_commit_group();
  }
}

// Write one 32 x 32 bf16 box (16 packed pairs per lane, lane = row) into a store
// box at `buf`, in the 64-byte-swizzled layout of the C tensor map.  The caller
// has waited until no TMA store still reads the box, and fences the async proxy
// from every writing thread before a store is issued on it (deepseek-ai/DeepGEMM
// PR 453, Fix: the fence is executed by all threads, not only the issuing one).
__device__ __forceinline__ void stage_box32(uint32_t buf, const uint32_t (&packed)[16], int lane) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    st_shared_v4(cbox_chunk_addr<32>(buf, lane, k), packed[4 * k], packed[4 * k + 1], packed[4 * k + 2],
                 packed[4 * k + 3]);
}

// bf16-round 32 fp32 values (given as bit patterns) into 16 packed pairs.
__device__ __forceinline__ void pack_row32(const uint32_t (&v)[32], uint32_t (&packed)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
    packed[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
}

// Same, after multiplying value j by row_scale and then by col_scale[j]
// (col_scale in shared memory, 8-byte aligned), two lanes per instruction.
__device__ __forceinline__ void scale_pack_row32(const uint32_t (&v)[32], float row_scale,
                                                 const float* col_scale, uint32_t (&packed)[16]) {
  const uint64_t rs = pack_f32x2(__float_as_uint(row_scale), __float_as_uint(row_scale));
  const uint64_t* cs = reinterpret_cast<const uint64_t*>(col_scale);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint64_t x = mul_f32x2(mul_f32x2(pack_f32x2(v[2 * j], v[2 * j + 1]), rs), cs[j]);
    float lo, hi;
    unpack_f32x2(x, lo, hi);
    packed[j] = pack_bf16x2(lo, hi);
  }
}

// Epilogue worker for one output tile, run by one warp on 32 rows (its TMEM lane
// quarter) and NCOLS columns starting at the accumulator address `taddr`.  Values
// are read from TMEM, multiplied by `row_scale * col_scale[c]` when SCALED,
// rounded to bf16 and stored through the warp's NBOX store boxes `bufs` (box
// counter `box`).  `release()` runs once, right after the last TMEM load.
template <int NCOLS, bool SCALED, int NBOX = 2, int W = 32, typename Release>
__device__ __forceinline__ void epilogue_tile(uint32_t taddr, uint32_t bufs, uint32_t& box,
                                              const float* col_scale, float row_scale,
                                              const CUtensorMap* tmC, int n_start, int m_start, int N,
                                              int M, int lane, Release&& release) {
  static_assert(NCOLS % 32 == 0, "epilogue works in 32-column steps");
  static_assert(W == 32 || NCOLS % 64 == 0, "64-column boxes need a multiple of 64 columns");
  auto convert = [&](const uint32_t (&v)[32], int cc, uint32_t* packed) {
    uint32_t (&pk)[16] = *reinterpret_cast<uint32_t(*)[16]>(packed);
    if constexpr (SCALED)
      scale_pack_row32(v, row_scale, col_scale + cc, pk);
    else
      pack_row32(v, pk);
  };
#pragma unroll 1
  for (int c = 0; c + 64 <= NCOLS; c += 64) {
    uint32_t v0[32], v1[32];
    tmem_ld_32x32b_x32(taddr + c, v0);
    tmem_ld_32x32b_x32(taddr + c + 32, v1);
    tmem_wait_ld();
    if (c + 64 == NCOLS) release();
    if constexpr (W == 64) {
      uint32_t packed[32];
      convert(v0, c, packed);
      convert(v1, c + 32, packed + 16);
      store_box<NBOX, 64>(bufs, box, packed, tmC, n_start + c, m_start, N, M, lane);
    } else {
      uint32_t packed[16];
      convert(v0, c, packed);
      store_box<NBOX, 32>(bufs, box, packed, tmC, n_start + c, m_start, N, M, lane);
      convert(v1, c + 32, packed);
      store_box<NBOX, 32>(bufs, box, packed, tmC, n_start + c + 32, m_start, N, M, lane);
    }
  }
  if constexpr (NCOLS % 64 == 32) {
    constexpr int c = NCOLS - 32;
    uint32_t v0[32];
    tmem_ld_32x32b_x32(taddr + c, v0);
    tmem_wait_ld();
    release();
    uint32_t packed[16];
    convert(v0, c, packed);
    store_box<NBOX, 32>(bufs, box, packed, tmC, n_start + c, m_start, N, M, lane);
  }
}

}  // namespace sg
