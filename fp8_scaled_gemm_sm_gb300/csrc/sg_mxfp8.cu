// sg_mxfp8.cu -- persistent block-scaled GEMM for the mxfp8 mode.
//
//   C[m,n] = bf16( sum_j acc_j[m,n] * 2^(sa[j][m]-127) * 2^(sb[j][n]-127) )
//
// with e4m3 operands and one e8m0 scale per 32 consecutive K elements of every
// row of A and of B (ROCm/mori PR 785, cost table and Scope: the "mxfp8" mode).
// The scales are applied inside the tensor core by
// tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X, which reads them from
// TMEM; nothing is rescaled in the epilogue.
//
// Per CTA (one per SM, persistent over 128 x 224 output tiles; 224 divides the
// 7168-wide weight exactly and leaves TMEM room for the scale factors next to
// two 224-column accumulators):
//   warp 0     TMA producer: A, B and the two raw scale boxes (sa rows
//              [4 K-blocks][128 m], sb rows [4][224 n], K-block major as they
//              sit in memory) into stage s; one full[s] barrier covers all four.
//   warp 1     TMEM owner and MMA issuer.  Per stage: wait sf_ready[s], copy the
//              stage's scale factors shared -> TMEM with two tcgen05.cp (128x128b
//              for A, 128x256b for B's two 128-row chunks), then 4 block-scaled
//              MMAs (K = 32 each, scale-factor id k selects the k-th byte of each
//              32-bit scale word), commit empty[s].
//   warp 2     scale-factor warp: wait full[s], regroup the raw bytes into the
//              layout the MMA reads (in every 32-lane quarter, lane r column c
//              holds the word for row 32 c + r of a 128-row chunk, each word the
//              four K-block scales of that row), fence the async proxy, arrive
//              sf_ready[s].  Its fence also orders its generic reads of the raw
//              boxes before the TMA refill of stage s (deepseek-ai/DeepGEMM PR 453,
//              Fix).
//   warps 3-6  epilogue: TMEM -> bf16 -> shared memory -> TMA store.
// Scale factors live in TMEM per stage (12 columns each), so a copy for stage s
// never overwrites scales that an MMA issued for an earlier stage still reads:
// the copy for a stage's next round is issued only after that stage's empty
// barrier, which tcgen05.commit fires once those MMAs have finished.
#include <cuda.h>
#include <cuda_runtime.h>

#include "sg_common.cuh"
#include "sg_internal.h"

namespace sg {

namespace {

constexpr int kMxBN = 224;
constexpr int kMxStages = 4;
constexpr int kMxEpiWarps = 4;
constexpr int kMxThreads = 96 + 32 * kMxEpiWarps;

struct MxLayout {
  static constexpr int kAStage = kBM * kRowBytes;        // 16 KB
  static constexpr int kBStage = kMxBN * kRowBytes;      // 28 KB
  static constexpr int kRawA = 4 * kBM;                  // [4][128] e8m0
  static constexpr int kRawB = 4 * kMxBN;                // [4][224] e8m0
  static constexpr int kSfA = 2048;                      // 128 lanes x 16 B
  static constexpr int kSfB = 4096;                      // 128 lanes x 32 B
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kMxStages * kAStage;
  static constexpr int kOffC = kOffB + kMxStages * kBStage;
  static constexpr int kOffRawA = kOffC + kMxEpiWarps * 2 * kCBoxBytes;
  static constexpr int kOffRawB = kOffRawA + kMxStages * kRawA;
  static constexpr int kOffSfA = kOffRawB + kMxStages * kRawB;
  static constexpr int kOffSfB = kOffSfA + kMxStages * kSfA;
  static constexpr int kOffBar = kOffSfB + kMxStages * kSfB;
  static constexpr int kNumBars = 3 * kMxStages + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 4 * kMxStages;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kOffB % 1024 == 0 && kOffC % 1024 == 0, "alignment");
  static_assert(kOffRawA % 128 == 0 && kOffRawB % 128 == 0 && kRawB % 128 == 0, "TMA alignment");
  static_assert(kOffSfA % 128 == 0 && kOffSfB % 128 == 0, "scale chunk alignment");
};

// TMEM columns: accumulators at 0 and 256 (224 wide each); per-stage scale
// factors in the gaps [224, 256) and [480, 512): A 4 columns, B 8 columns.
__device__ __forceinline__ uint32_t sf_col_a(int s) { return s < 2 ? 224 + 12 * s : 480 + 12 * (s - 2); }
__device__ __forceinline__ uint32_t sf_col_b(int s) { return sf_col_a(s) + 4; }

// Scale factors go to TMEM with two copies per stage: tcgen05.cp.128x128b for A
// (lane l, columns 0-3) and tcgen05.cp.128x256b for B (lane l, columns 0-7).
// For a 128-row chunk the MMA takes, in every 32-lane quarter, lane r and column
// c to hold the four K-block scales (bytes 0-3) of row 32 c + r of the chunk.
// The shared-memory source is therefore the same 16 (A) or 32 (B) bytes for
// lanes r, r+32, r+64, r+96, laid out in 8-row x 16-byte core matrices:
// row l, 16-byte chunk j at (l / 8) * SBO + j * LBO + (l % 8) * 16.
__device__ __forceinline__ uint64_t sf_desc_a(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }
__device__ __forceinline__ uint64_t sf_desc_b(uint32_t addr) { return smem_desc(addr, 128, 256, 0); }

__device__ __forceinline__ void tmem_cp_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// The four 32-bit scale words lane r contributes for a 128-row chunk starting at
// row0 of a raw K-block-major box ([4 K blocks][pitch] e8m0 bytes): word w holds
// the 4 K-block scales of row row0 + 32 w + r (0 past rows_valid).
__device__ __forceinline__ void sf_words(const uint8_t* raw, int pitch, int row0, int rows_valid, int lane,
                                         uint32_t (&w)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int row = row0 + 32 * q + lane;
    uint32_t v = 0;
    if (row < rows_valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v |= static_cast<uint32_t>(raw[k * pitch + row]) << (8 * k);
    }
    w[q] = v;
  }
}

__global__ void __launch_bounds__(kMxThreads, 1)
    mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                      const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using L = MxLayout;
  constexpr int kBK = 128;
  constexpr int kKSteps = 4;
  constexpr uint32_t kTx = L::kAStage + L::kBStage + L::kRawA + L::kRawB;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kAccStride = 256;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem + L::kOffA);
  const uint32_t sB = smem_addr(smem + L::kOffB);
  const uint32_t sC = smem_addr(smem + L::kOffC);
  const uint32_t sRawA = smem_addr(smem + L::kOffRawA);
  const uint32_t sRawB = smem_addr(smem + L::kOffRawB);
  const uint32_t sSfA = smem_addr(smem + L::kOffSfA);
  const uint32_t sSfB = smem_addr(smem + L::kOffSfB);
  const uint32_t bar0 = smem_addr(smem + L::kOffBar);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kMxStages + s); };
  auto sf_bar = [&](int s) { return bar0 + 8 * (2 * kMxStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8 * (3 * kMxStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8 * (3 * kMxStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8 * (3 * kMxStages + 4);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  uint32_t* last_par = misc + 4;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 32 * kMxEpiWarps);
    }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const Watchdog wd{p.status, p.timeout_ns, reinterpret_cast<volatile int*>(&misc[1])};

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
      int stage = 0, kstep = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = tile_coord(p, t);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          if (kstep != p.skip_kstep) {
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, kTx);
            tma_load_2d(sA + stage * L::kAStage, &tmA, kb * kBK, tc.mb * kBM, fb);
            tma_load_2d(sB + stage * L::kBStage, &tmB, kb * kBK, tc.nb * kMxBN, fb);
            tma_load_2d(sRawA + stage * L::kRawA, &tmSA, tc.mb * kBM, kb * 4, fb);
            tma_load_2d(sRawB + stage * L::kRawB, &tmSB, tc.nb * kMxBN, kb * 4, fb);
            issued |= 1u << stage;
            last_par[stage] = phase;
          }
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < kMxStages; ++s)
          if ((issued >> s) & 1) mbar_wait_drain(full_bar(s), last_par[s], 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------- scale-factor copies + MMA issuer ----------------
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait(tempty_bar(acc), acc_par ^ 1, wd, kWhereMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccStride;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, wd, kWhereMmaFull) ||
              !mbar_wait(sf_bar(stage), phase, wd, kWhereMmaSf)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tsa = tmem_base + sf_col_a(stage);
          const uint32_t tsb = tmem_base + sf_col_b(stage);
          tmem_cp_128x128b(tsa, sf_desc_a(sSfA + stage * L::kSfA));
          tmem_cp_128x256b(tsb, sf_desc_b(sSfB + stage * L::kSfB));
          const uint32_t a0 = sA + stage * L::kAStage;
          const uint32_t b0 = sB + stage * L::kBStage;
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {
            mma_mxf8(d, kmajor_sw128_desc(a0 + 32 * k), kmajor_sw128_desc(b0 + 32 * k),
                     instr_desc_mx(kBM, kMxBN, k, k), tsa, tsb, (kb | k) != 0);
          }
          mma_commit(empty_bar(stage));
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
      }
      if (!ok) {
        mma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else if (warp == 2) {
    // ---------------- scale-factor regrouping ----------------
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      bool ok = true;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        ok = mbar_wait(full_bar(stage), phase, wd, kWhereSfFull);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const uint8_t* rawA = smem + L::kOffRawA + stage * L::kRawA;
        const uint8_t* rawB = smem + L::kOffRawB + stage * L::kRawB;
        uint32_t wa[4], wb0[4], wb1[4];
        sf_words(rawA, kBM, 0, kBM, lane, wa);
        sf_words(rawB, kMxBN, 0, kMxBN, lane, wb0);
        sf_words(rawB, kMxBN, 128, kMxBN, lane, wb1);
        const uint32_t dA = sSfA + stage * L::kSfA;
        const uint32_t dB = sSfB + stage * L::kSfB;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // the same words for lanes r + 32 q
          const int l = 32 * q + lane;
          st_shared_v4(dA + (l >> 3) * 128 + (l & 7) * 16, wa[0], wa[1], wa[2], wa[3]);
          st_shared_v4(dB + (l >> 3) * 256 + (l & 7) * 16, wb0[0], wb0[1], wb0[2], wb0[3]);
          st_shared_v4(dB + (l >> 3) * 256 + 128 + (l & 7) * 16, wb1[0], wb1[1], wb1[2], wb1[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_bar(stage));
        if (++stage == kMxStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp - 3;
    const int quarter = warp & 3;
    const uint32_t bufs = sC + ew * 2 * kCBoxBytes;
    int it = 0;
    uint32_t box = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const TileCoord tc = tile_coord(p, t);
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      const int m_start = tc.mb * kBM + quarter * 32;
      const int n_start = tc.nb * kMxBN;
      const bool ok = mbar_wait(tfull_bar(acc), acc_par, wd, kWhereEpiTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccStride;
      epilogue_tile<kMxBN, false>(taddr, bufs, box, nullptr, 0.f, &tmC, n_start, m_start, p.N, p.M,
                                  lane, [&]() {
                                    tc_fence_before();
                                    mbar_arrive(tempty_bar(acc));
                                  });
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t mxfp8_prepare() {
  return cudaFuncSetAttribute(mxfp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MxLayout::kDynSmem);
}

sg_status_t mxfp8_launch(const LaunchArgs& a) {
  CUtensorMap tmA, tmB, tmSA, tmSB, tmC;
  const uint64_t kblk = static_cast<uint64_t>(a.K / 32);
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, 128, kBM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.K, a.N, a.K, 128, kMxBN,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmSA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_scale, a.M, kblk, a.M, kBM, 4,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tmSB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_scale, a.N, kblk, a.N, kMxBN, 4,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.N, a.M, a.N * 2, kCBoxCols, kCBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return SG_ERR_CUDA;
  GemmParams p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.m_blocks = static_cast<int32_t>((a.M + kBM - 1) / kBM);
  p.n_blocks = static_cast<int32_t>((a.N + kMxBN - 1) / kMxBN);
  p.k_blocks = static_cast<int32_t>((a.K + 127) / 128);
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.skip_kstep = a.skip_kstep;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  const int grid = p.num_tiles < a.num_sms ? p.num_tiles : a.num_sms;
  mxfp8_gemm_kernel<<<grid, kMxThreads, MxLayout::kDynSmem, a.stream>>>(tmA, tmB, tmSA, tmSB, tmC, p);
  return launch_status();
}

void mxfp8_config(TileConfig* c) {
  c->bm = kBM;
  c->bn = kMxBN;
  c->bk = 128;
  c->stages = kMxStages;
}

}  // namespace sg
