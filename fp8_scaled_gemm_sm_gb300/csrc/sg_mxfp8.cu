// sg_mxfp8.cu -- persistent block-scaled GEMM for the mxfp8 mode.
//
//   C[m,n] = bf16( sum_j acc_j[m,n] * 2^(sa[j][m]-127) * 2^(sb[j][n]-127) )
//
// with e4m3 operands and one e8m0 scale per 32 consecutive K elements of every
// row of A and of B (ROCm/mori PR 785, cost table and Scope: the "mxfp8" mode).
// The scales are applied inside the tensor core by
// tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X, which reads
// them from TMEM; nothing is rescaled in the epilogue.
//
// Two kernels per launch:
//
// 1. mx_scale_records_kernel rearranges the scales, which arrive K-block major
//    ([K/32][M] and [K/32][N] bytes, ROCm/mori PR 809, Not done yet), into
//    records in the plan's workspace.  The MMA expects, in every 32-lane quarter
//    of TMEM, lane r column c to hold the four K-block scales of row 32 c + r of
//    a 128-row chunk.  A: one 512-byte record per 128-row chunk and 128-element
//    K step, byte 16 r + 4 c + k = the scale of row 32 c + r for the step's K
//    block k: the source tcgen05.cp.32x128b.warpx4 copies (32 lanes x 16 bytes,
//    repeated by the copy into all four lane quarters).  B: one 4 KB record per
//    224-row N tile and K step holding both of the tile's 128-row chunks for all
//    128 lanes (already repeated per quarter): the source of a single
//    tcgen05.cp.128x256b, so a stage needs two copies, not three (measured 5%
//    faster).  Missing rows and K blocks are 0 (their A / B values are
//    zero-filled by TMA).  It reads (M + N) K / 32 bytes and writes (M + 4 N) K / 32.
//
// 2. mxfp8_pair_kernel<224>: two CTAs on neighbouring SMs (a cluster of 2) compute
//    one 256 x 224 output tile with the pair MMA.  Each CTA stages its own 128
//    rows of A and 112 of the tile's 224 rows of B, so per SM the shared memory
//    written by TMA and read by the MMA per FLOP is that of a 128 x 448 tile; a
//    single-CTA 128 x 224 tile was bound by that traffic (44 KB written and
//    44 KB read per 470-cycle stage).  224 divides the 7168-wide weight exactly
//    and leaves TMEM room for the scale factors next to two 224-column
//    accumulators.  The scale records travel with the operands: per stage each
//    CTA loads its A record and the tile's B record by TMA, and all of it
//    completes the even CTA's full[s].  (Regrouping the raw scales in a warp of
//    each CTA instead put a per-stage cross-CTA release on the critical path and
//    ran 2x slower.)
//
//    mxfp8_pair_kernel<128> is the same kernel on 256 x 128 tiles, for launches
//    where 224-wide tiles would leave pairs of SMs idle (small M); its B scales
//    fit one 128-row chunk and travel in 512-byte records like A's.
//
// Per CTA of the pair kernel, persistent over pair tiles (N block fastest):
//   warp 0     TMA producer: A rows, B half and scale records into stage s.
//   warp 1     TMEM owner (both CTAs) and, in the even CTA, MMA issuer.  Per
//              stage: wait full[s]; copy both CTAs' scale records to TMEM with
//              tcgen05.cp.cta_group::2 (each CTA's copy reads its own shared
//              memory): 32x128b.warpx4 for A's chunk, 128x256b for B's two
//              chunks; 4 pair MMAs (K = 32 each; scale-factor id k selects the
//              k-th byte of each 32-bit scale word); commit empty[s] of both CTAs.
//   warps 2-9  epilogue, two warps per TMEM lane quarter (columns 0-127 and
//              128-223): TMEM -> bf16 -> shared memory -> TMA store; the release
//              of an accumulator arrives on the even CTA's tmem_empty.
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

constexpr int kMxBN = 224;                 // N of a wide pair tile (and of each CTA's accumulator)
constexpr int kMxBNarrow = 128;            // N of a narrow pair tile
constexpr int kMxEpiWarps = 8;
constexpr int kMxThreads = 64 + 32 * kMxEpiWarps;
constexpr int kRec = 512;                  // bytes of one scale record (32 rows x 16 B)

// The two tile widths.  Wide (224): B's scales span two 128-row chunks, held in
// one 4 KB record per tile and K step (one 128x256b copy); 5 stages.  Narrow
// (128): one chunk, held like A's in a 512-byte record (one 32x128b.warpx4 copy);
// B stages are half as large, so 6 stages fit.
template <int BN>
struct MxTile {
  static_assert(BN == kMxBN || BN == kMxBNarrow, "tile width");
  static constexpr bool kWide = BN == kMxBN;
  static constexpr int kBHalf = BN / 2;    // B rows each CTA stages
  static constexpr int kStages = kWide ? 5 : 6;
  static constexpr int kSfB = kWide ? 8 * kRec : kRec;
  static constexpr int kSfBRows = kSfB / kRec;  // 512-byte record rows per B record
};

template <int BN>
struct MxLayout {
  using T = MxTile<BN>;
  static constexpr int kStages = T::kStages;
  static constexpr int kAStage = kBM * kRowBytes;        // 16 KB
  static constexpr int kBStage = T::kBHalf * kRowBytes;  // 14 KB (wide), 8 KB (narrow)
  static constexpr int kSfA = kRec;                      // A's record
  static constexpr int kSfB = T::kSfB;                   // B's record
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kAStage;
  static constexpr int kOffC = kOffB + kStages * kBStage;
  static constexpr int kOffSfA = kOffC + kMxEpiWarps * 2 * kCBoxBytes;
  static constexpr int kOffSfB = kOffSfA + kStages * kSfA;
  static constexpr int kOffBar = kOffSfB + kStages * kSfB;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 4 * kStages;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kOffB % 1024 == 0 && kBStage % 1024 == 0 && kOffC % 1024 == 0, "alignment");
  static_assert(kOffSfA % 128 == 0 && kOffSfB % 128 == 0, "TMA / scale-record alignment");
  static_assert(kDynSmem <= 232448, "shared memory");
};

// TMEM columns.  Wide: accumulators at 0 and 256 (224 wide each); per-stage scale
// factors (A 4 columns, B 8) in the gaps [224, 256) and [480, 512).  Narrow:
// accumulators at 0 and 256 (128 wide each); stage s's scale factors (A 4
// columns, B 4) at 128 + 8 s.
template <int BN>
__device__ __forceinline__ uint32_t sf_col_a(int s) {
  if constexpr (BN == kMxBN) return s == 0 ? 224 : s == 1 ? 236 : s == 2 ? 480 : s == 3 ? 492 : 248;
  else return 128 + 8 * s;
}
template <int BN>
__device__ __forceinline__ uint32_t sf_col_b(int s) {
  if constexpr (BN == kMxBN) return s == 0 ? 228 : s == 1 ? 240 : s == 2 ? 484 : s == 3 ? 496 : 504;
  else return 132 + 8 * s;
}
static_assert(MxTile<kMxBN>::kStages <= 5, "TMEM has scale-factor room for 5 wide stages");
static_assert(128 + 8 * MxTile<kMxBNarrow>::kStages <= 256, "narrow scale factors below the second accumulator");

// A 32-row x 16-byte record in shared memory as 8-row x 16-byte core matrices:
// row r at (r / 8) * 128 + (r % 8) * 16 = 16 r.
__device__ __forceinline__ uint64_t rec_desc(uint32_t addr) { return smem_desc(addr, 0, 128, 0); }

__device__ __forceinline__ void tmem_cp_pair_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Records of the workspace, in 512-byte rows.  A: record (mc, ks) is row
// mc * k_steps + ks.  B, wide tiles: the record of (N tile nt, step ks) is 8 rows
// from row (nt * k_steps + ks) * 8: the 128-lane x 32-byte source of one
// tcgen05.cp.128x256b, lane l holding its 16-byte words for the tile's 128-row
// chunks 0 and 1 at (l / 8) * 256 + j * 128 + (l % 8) * 16 (every 32-lane quarter
// repeats the same rows, as the MMA wants them in every quarter).  B, narrow
// tiles: row nt * k_steps + ks, laid out as A's records.
struct RecGeom {
  int M, N, kblk, k_steps, m_chunks, n_tiles;
  bool wide;  // B records for 224-row tiles (else 128-row tiles)
  __host__ __device__ int64_t a_records() const { return static_cast<int64_t>(m_chunks) * k_steps; }
  __host__ __device__ int64_t b_rows() const {
    return static_cast<int64_t>(n_tiles) * k_steps * (wide ? 8 : 1);
  }
};

// One thread per 32-bit word: the four K-block scales of one row.  In an A record
// thread t handles row 32 c + r with r = t % 32, c = t / 32, so consecutive
// threads read consecutive bytes of each K-block row of the source.
__global__ void __launch_bounds__(256)
    mx_scale_records_kernel(const uint8_t* __restrict__ sa, const uint8_t* __restrict__ sb,
                            uint32_t* __restrict__ rec_a, uint32_t* __restrict__ rec_b, RecGeom g) {
  grid_dep_launch();
  grid_dep_wait();  // the previous GEMM may still read the records this kernel rewrites
  const int64_t words_a = g.a_records() * 128;
  const int64_t words_b = g.b_rows() * 128;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < words_a + words_b;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_a = i < words_a;
    int row, ks, pitch;
    int64_t pos;  // word position in rec_a / rec_b
    const uint8_t* src;
    bool valid;
    if (is_a) {
      const int64_t rec = i >> 7;
      const int t = static_cast<int>(i & 127);
      const int r = t & 31, c = t >> 5;
      const int mc = static_cast<int>(rec / g.k_steps);
      ks = static_cast<int>(rec - static_cast<int64_t>(mc) * g.k_steps);
      row = mc * kBM + 32 * c + r;
      valid = row < g.M;
      src = sa;
      pitch = g.M;
      pos = rec * 128 + r * 4 + c;
    } else if (g.wide) {
      const int64_t wi = i - words_a;
      const int64_t q = wi >> 10;  // (nt, ks) record: 1024 words
      const int t = static_cast<int>(wi & 1023);
      const int l = t >> 3, j = (t >> 2) & 1, c = t & 3;  // lane, 128-row chunk, word
      const int nt = static_cast<int>(q / g.k_steps);
      ks = static_cast<int>(q - static_cast<int64_t>(nt) * g.k_steps);
      const int local = 128 * j + 32 * c + (l & 31);  // row within the 224-row tile
      row = nt * kMxBN + local;
      valid = local < kMxBN && row < g.N;
      src = sb;
      pitch = g.N;
      pos = q * 1024 + (l >> 3) * 64 + j * 32 + (l & 7) * 4 + c;
    } else {
      const int64_t wi = i - words_a;
      const int64_t q = wi >> 7;  // (nt, ks) record: 128 words, as A's
      const int t = static_cast<int>(wi & 127);
      const int r = t & 31, c = t >> 5;
      const int nt = static_cast<int>(q / g.k_steps);
      ks = static_cast<int>(q - static_cast<int64_t>(nt) * g.k_steps);
      row = nt * kMxBNarrow + 32 * c + r;
      valid = row < g.N;
      src = sb;
      pitch = g.N;
      pos = q * 128 + r * 4 + c;
    }
    uint32_t w = 0;
    if (valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int kb = 4 * ks + k;
        if (kb < g.kblk) w |= static_cast<uint32_t>(__ldg(src + static_cast<int64_t>(kb) * pitch + row)) << (8 * k);
      }
    }
    (is_a ? rec_a : rec_b)[pos] = w;
  }
}

__device__ __forceinline__ void tmem_cp_pair_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int BN>
__global__ void __launch_bounds__(kMxThreads, 1)
    mxfp8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmRA, const __grid_constant__ CUtensorMap tmRB,
                      const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using L = MxLayout<BN>;
  using T = MxTile<BN>;
  constexpr int kMxStages = L::kStages;
  constexpr int kBK = 128;
  constexpr int kKSteps = 4;
  constexpr uint32_t kTxPair = 2 * (L::kAStage + L::kBStage + L::kSfA + L::kSfB);  // both CTAs' bytes
  constexpr uint32_t kTmemCols = 512;
  constexpr int kAccStride = 256;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem + L::kOffA);
  const uint32_t sB = smem_addr(smem + L::kOffB);
  const uint32_t sC = smem_addr(smem + L::kOffC);
  const uint32_t sSfA = smem_addr(smem + L::kOffSfA);
  const uint32_t sSfB = smem_addr(smem + L::kOffSfB);
  const uint32_t bar0 = smem_addr(smem + L::kOffBar);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kMxStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8 * (2 * kMxStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8 * (2 * kMxStages + 2 + a); };
  const uint32_t drain_bar = bar0 + 8 * (2 * kMxStages + 4);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  uint32_t* last_par = misc + 4;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_cta_rank());
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(num_clusters_x());
  const int num_pair_tiles = ((p.M + 2 * kBM - 1) / (2 * kBM)) * p.n_blocks;
  auto coord = [&](int tp) {
    TileCoord c;
    const int mp = tp / p.n_blocks;
    c.nb = tp - mp * p.n_blocks;
    c.mb = 2 * mp + rank;  // this CTA's 128-row block (past M: zero rows, clipped stores)
    return c;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(full_bar(s), 1);   // the even CTA's producer arms it for both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // one pair commit per round
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * 32 * kMxEpiWarps);  // both CTAs' epilogue threads
    }
    mbar_init(drain_bar, 1);
    misc[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates together
    tmem_alloc_pair(smem_addr(&misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const Watchdog wd{p.status, p.timeout_ns, reinterpret_cast<volatile int*>(&misc[1])};
  grid_dep_launch();
  grid_dep_wait();  // no global memory is touched before this point

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint64_t keep_b = l2_policy_evict_last();
      tma_prefetch_desc(&tmRA);
      tma_prefetch_desc(&tmRB);
      int stage = 0, kstep = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs) {
        const TileCoord tc = coord(tp);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
          if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          if (kstep != p.skip_kstep) {
            const uint32_t fb = map_to_cta(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), kTxPair);
            tma_load_2d_pair(sA + stage * L::kAStage, &tmA, kb * kBK, tc.mb * kBM, fb);
            tma_load_2d_pair_hint(sB + stage * L::kBStage, &tmB, kb * kBK, tc.nb * BN + rank * T::kBHalf, fb,
                                  keep_b);
            // records past the last M chunk read as zeros
            tma_load_2d_pair(sSfA + stage * L::kSfA, &tmRA, 0, tc.mb * p.k_blocks + kb, fb);
            tma_load_2d_pair(sSfB + stage * L::kSfB, &tmRB, 0, (tc.nb * p.k_blocks + kb) * T::kSfBRows, fb);
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
        if (leader) {
          for (int s = 0; s < kMxStages; ++s)
            if ((issued >> s) & 1) mbar_wait_drain(full_bar(s), last_par[s], 200000000ull);
        } else {
          // this CTA's loads complete on the even CTA's barrier: give them time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 2000000ull) {
          }
        }
      } else {
        // every pair commit to this CTA's empty barriers must land before exit
        for (int s = 0; s < kMxStages; ++s)
          if ((issued >> s) & 1) mbar_wait_drain(empty_bar(s), last_par[s], 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------- scale-factor copies + pair MMA issuer (even CTA) ----------------
    if (lane == 0 && leader) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint64_t desc_a = kmajor_sw128_desc(sA), desc_b = kmajor_sw128_desc(sB);
      const uint64_t desc_sfa = rec_desc(sSfA);
      const uint64_t desc_sfb = T::kWide ? smem_desc(sSfB, 128, 256, 0) : rec_desc(sSfB);
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait_cluster(tempty_bar(acc), acc_par ^ 1, wd, kWhereMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccStride;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_cluster(full_bar(stage), phase, wd, kWhereMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tsa = tmem_base + sf_col_a<BN>(stage);
          const uint32_t tsb = tmem_base + sf_col_b<BN>(stage);
          tmem_cp_pair_32x128b_x4(tsa, desc_advance(desc_sfa, stage * L::kSfA));
          if constexpr (T::kWide)
            tmem_cp_pair_128x256b(tsb, desc_advance(desc_sfb, stage * L::kSfB));
          else
            tmem_cp_pair_32x128b_x4(tsb, desc_advance(desc_sfb, stage * L::kSfB));
          const uint64_t da = desc_advance(desc_a, stage * L::kAStage);
          const uint64_t db = desc_advance(desc_b, stage * L::kBStage);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {
            mma_mxf8_pair(d, desc_advance(da, 32 * k), desc_advance(db, 32 * k),
                          instr_desc_mx(2 * kBM, BN, k, k), tsa, tsb, (kb | k) != 0);
          }
          mma_commit_pair_both(empty_bar(stage));
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(tfull_bar(acc));
      }
      if (!ok) {  // let issued MMAs finish before TMEM is freed
        mma_commit_pair(drain_bar);
        mbar_wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int ew = warp - 2;                 // 0 .. 7
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    // wide: columns 0-127 or 128-223 of the tile; narrow: 0-63 or 64-127
    constexpr int kColsLo = T::kWide ? 128 : 64;
    constexpr int kColsHi = BN - kColsLo;
    const int col0 = ew < 4 ? 0 : kColsLo;
    const uint32_t bufs = sC + ew * 2 * kCBoxBytes;
    int it = 0;
    uint32_t box = 0;
    for (int tp = pair; tp < num_pair_tiles; tp += npairs, ++it) {
      const TileCoord tc = coord(tp);
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      const int m_start = tc.mb * kBM + quarter * 32;
      const int n_start = tc.nb * BN + col0;
      const bool ok = mbar_wait_cluster(tfull_bar(acc), acc_par, wd, kWhereEpiTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kAccStride + col0;
      const uint32_t release_bar = map_to_cta(tempty_bar(acc), 0);
      auto release = [&]() {
        tc_fence_before();
        mbar_arrive_cluster_relaxed(release_bar);
      };
      if (ew < 4)
        epilogue_tile<kColsLo, false>(taddr, bufs, box, nullptr, 0.f, &tmC, n_start, m_start, p.N, p.M, lane,
                                      release);
      else
        epilogue_tile<kColsHi, false>(taddr, bufs, box, nullptr, 0.f, &tmC, n_start, m_start, p.N, p.M, lane,
                                      release);
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it or use its TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

RecGeom rec_geom(int64_t M, int64_t N, int64_t K, int bn) {
  RecGeom g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.kblk = static_cast<int>(K / 32);
  g.k_steps = static_cast<int>((K + 127) / 128);
  g.m_chunks = static_cast<int>((M + kBM - 1) / kBM);
  g.n_tiles = static_cast<int>((N + bn - 1) / bn);
  g.wide = bn == kMxBN;
  return g;
}

// Tile width of a launch: the one with the smaller estimate of waves of pair
// tiles x tile width x cost of a column.  A narrow tile's column costs more (it
// stages A once per 128 columns instead of per 224, and copies two scale records
// per 128 columns): 1.32-1.42x, from timings at N = 7168, K = 1792 and M = 2048
// to 8192.  Narrow tiles win where wide ones leave pairs idle: at M = 256 (one
// row of 32 wide tiles on 76 pairs) 21-22 us against 24-25 us.
constexpr double kNarrowColumnCost = 1.4;

int tile_bn_for(int64_t M, int64_t N, int num_sms, int pinned) {
  if (pinned) return pinned;
  const int64_t pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const int64_t mp = (M + 2 * kBM - 1) / (2 * kBM);
  const int64_t tiles_w = mp * ((N + kMxBN - 1) / kMxBN);
  const int64_t tiles_n = mp * ((N + kMxBNarrow - 1) / kMxBNarrow);
  const double est_w = static_cast<double>((tiles_w + pairs - 1) / pairs) * kMxBN;
  const double est_n = static_cast<double>((tiles_n + pairs - 1) / pairs) * kMxBNarrow * kNarrowColumnCost;
  return est_n < est_w ? kMxBNarrow : kMxBN;
}

template <int BN>
sg_status_t launch_pair(const LaunchArgs& a, const RecGeom& g, const uint32_t* rec_a, const uint32_t* rec_b) {
  using T = MxTile<BN>;
  CUtensorMap tmA, tmB, tmRA, tmRB, tmC;
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, 128, kBM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.K, a.N, a.K, 128, T::kBHalf,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmRA, CU_TENSOR_MAP_DATA_TYPE_UINT32, rec_a, kRec / 4, g.a_records(), kRec, kRec / 4, 1,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tmRB, CU_TENSOR_MAP_DATA_TYPE_UINT32, rec_b, kRec / 4, g.b_rows(), kRec, kRec / 4,
                 T::kSfBRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.N, a.M, a.N * 2, kCBoxCols, kCBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return SG_ERR_CUDA;
  GemmParams p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.m_blocks = static_cast<int32_t>((a.M + kBM - 1) / kBM);
  p.n_blocks = static_cast<int32_t>((a.N + BN - 1) / BN);
  p.k_blocks = static_cast<int32_t>((a.K + 127) / 128);
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.skip_kstep = a.skip_kstep;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  const int pair_tiles = static_cast<int>((a.M + 2 * kBM - 1) / (2 * kBM)) * p.n_blocks;
  const int max_pairs = a.num_sms / 2;
  const int pairs = pair_tiles < max_pairs ? pair_tiles : max_pairs;
  GemmLaunch l(dim3(pairs * 2), dim3(kMxThreads), MxLayout<BN>::kDynSmem, a.stream, 2);
  const cudaError_t e = cudaLaunchKernelEx(&l.cfg, mxfp8_pair_kernel<BN>, tmA, tmB, tmRA, tmRB, tmC, p);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();  // clear the non-sticky launch error
    return SG_ERR_CUDA;
  }
  return SG_OK;
}

}  // namespace

// Both widths' records fit: the wide tiles' B records (8 rows per 224 columns)
// outnumber the narrow tiles' (1 row per 128 columns) for every N.
size_t mxfp8_workspace_bytes(int64_t M_max, int64_t N, int64_t K) {
  const RecGeom g = rec_geom(M_max, N, K, kMxBN);
  return static_cast<size_t>(g.a_records() + g.b_rows()) * kRec;
}

cudaError_t mxfp8_prepare() {
  const cudaError_t e = cudaFuncSetAttribute(mxfp8_pair_kernel<kMxBN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             MxLayout<kMxBN>::kDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mxfp8_pair_kernel<kMxBNarrow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MxLayout<kMxBNarrow>::kDynSmem);
}

bool mxfp8_tile_ok(int bn) { return bn == kMxBN || bn == kMxBNarrow; }

sg_status_t mxfp8_launch(const LaunchArgs& a) {
  const int bn = tile_bn_for(a.M, a.N, a.num_sms, a.tile_bn);
  const RecGeom g = rec_geom(a.M, a.N, a.K, bn);
  // B's records first: their count depends on N, K and the width only, so A's
  // (which grow with M) never overlap them.
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  uint32_t* rec_b = reinterpret_cast<uint32_t*>(ws);
  uint32_t* rec_a = reinterpret_cast<uint32_t*>(ws + g.b_rows() * kRec);
  {
    const int64_t words = (g.a_records() + g.b_rows()) * 128;
    const int64_t blocks = (words + 255) / 256;
    const int grid = static_cast<int>(blocks < 4L * a.num_sms * 8 ? blocks : 4L * a.num_sms * 8);
    GemmLaunch l(dim3(grid), dim3(256), 0, a.stream, 1);
    const cudaError_t e = cudaLaunchKernelEx(&l.cfg, mx_scale_records_kernel, static_cast<const uint8_t*>(a.a_scale),
                                             static_cast<const uint8_t*>(a.b_scale), rec_a, rec_b, g);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();  // clear the non-sticky launch error
      return SG_ERR_CUDA;
    }
  }
  return bn == kMxBN ? launch_pair<kMxBN>(a, g, rec_a, rec_b) : launch_pair<kMxBNarrow>(a, g, rec_a, rec_b);
}

void mxfp8_config(int64_t M, int64_t N, int num_sms, int tile_bn, TileConfig* c) {
  const int bn = tile_bn_for(M, N, num_sms, tile_bn);
  c->bm = kBM;
  c->bn = bn;
  c->bk = 128;
  c->stages = bn == kMxBN ? MxTile<kMxBN>::kStages : MxTile<kMxBNarrow>::kStages;
  c->cluster = 2;
  c->rows_per_group = 2 * kBM;
}

}  // namespace sg
