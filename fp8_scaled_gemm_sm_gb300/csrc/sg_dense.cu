// sg_dense.cu -- persistent warp-specialised GEMM for the ptpc and bf16 modes.
//
//   C[m,n] = bf16(acc[m,n] * a_scale[m] * b_scale[n])   (ptpc, e4m3 x e4m3)
//   C[m,n] = bf16(acc[m,n])                             (bf16 x bf16)
//
// Every K runs on CTA pairs (a cluster of two CTAs on neighbouring SMs), each
// pair persistent over 256 x BN output tiles computed with the pair MMA
// (tcgen05.mma.cta_group::2); BN is 256, or 128 for launches with fewer 256-wide
// tiles than pairs of SMs, and a ragged last N block runs its MMAs only as wide as
// its remaining columns.  Per CTA:
//   warp 0      TMA producer: waits empty[s], loads this CTA's A rows [128 x
//               128 B] and its half of the tile's B rows [BN/2 x 128 B] (128-byte
//               swizzle) into stage s; the bytes of both CTAs complete the even
//               CTA's full[s], which its producer arms.
//   warp 1      allocates TMEM with the peer (two BN-column fp32 accumulators);
//               in the even CTA one thread waits full[s], issues 4 pair MMAs
//               (K = 32 fp8 / 16 bf16 each) and commits to empty[s] of both
//               CTAs, so a stage is handed back only after the tensor cores have
//               finished reading it; after a tile's last K block it commits to
//               tmem_full[acc] of both CTAs.
//   warps 2..   epilogue: wait tmem_full[acc], read this CTA's 128 accumulator
//               rows with tcgen05.ld, scale, round to bf16, stage in shared
//               memory, fence the async proxy, store by TMA; hand the
//               accumulator back with tcgen05.fence::before_thread_sync + an
//               arrive on the even CTA's tmem_empty[acc].
// A gather variant (ptpc, one CTA per SM, A rows gathered by index) follows.
//
// The stage / phase counters run continuously across tiles, so a K loop of one
// or two blocks (the "peeled tail" case, K <= 256) goes through exactly the
// same waits as a long one: no read of a stage happens before the wait on the
// barrier that its producer's bytes complete (ROCm/mori PR 785, Problem and
// Fix; ROCm/aiter PR 6539, Technical Details).  Stages are released only by
// tcgen05.commit, which fires after the MMAs that read them
// (deepseek-ai/DeepGEMM PR 453, ds-review-bot v4: "release smem only after
// UMMA commits").  The epilogue's generic shared-memory writes are fenced into
// the async proxy by every writing thread before the TMA store is issued
// (deepseek-ai/DeepGEMM PR 453, Fix).  No TMA load here is multicast: every
// CTA loads its own operand rows from this GPU's memory.  Each kernel touches
// global memory only after griddepcontrol.wait (programmatic dependent launch:
// the launch may begin while the previous kernel in the stream finishes).
#include <cuda.h>
#include <cuda_runtime.h>

#include "sg_common.cuh"
#include "sg_internal.h"

namespace sg {

// ---------------------------------------------------------------------------
// Pair kernel: two CTAs on neighbouring SMs compute one 256 x BN tile with
// tcgen05.mma.cta_group::2.  Each CTA stages its own 128 rows of A and its half
// (BN/2 rows) of B, so per SM the shared-memory operand traffic per FLOP is that
// of a 128 x 2BN tile; the even CTA of the pair issues the MMAs, the TMA bytes
// of both CTAs complete its full[s] barrier, its commits arrive on both CTAs'
// empty[s] and tmem_full[acc], and both CTAs' epilogues release the accumulator
// on its tmem_empty[acc].  Each CTA reads its own 128 accumulator rows.
// ---------------------------------------------------------------------------

template <int BN, int STAGES, int EPI_WARPS, int NBOX, int BOXW>
struct PairLayout {
  static constexpr int kAStage = kBM * kRowBytes;
  static constexpr int kBStage = (BN / 2) * kRowBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kAStage;
  static constexpr int kOffC = kOffB + STAGES * kBStage;
  static constexpr int kColsPerWarp = BN * 4 / EPI_WARPS;
  static constexpr int kOffScale = kOffC + EPI_WARPS * NBOX * cbox_bytes<BOXW>();
  static constexpr int kOffBar = kOffScale + EPI_WARPS * kColsPerWarp * 4;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 4 * STAGES;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kOffB % 1024 == 0 && kOffC % 1024 == 0, "alignment");
  static_assert(kDynSmem <= 232448, "shared memory");
};

template <int MODE, int BN, int STAGES, int EPI_WARPS, int NBOX, int BOXW>
__global__ void __launch_bounds__(64 + 32 * EPI_WARPS, 1)
    dense_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using L = PairLayout<BN, STAGES, EPI_WARPS, NBOX, BOXW>;
  constexpr bool kScaled = (MODE == kModePtpc);
  constexpr int kBK = (MODE == kModeBf16) ? 64 : 128;
  constexpr int kUmmaK = (MODE == kModeBf16) ? 16 : 32;
  constexpr int kKSteps = kBK / kUmmaK;
  constexpr uint32_t kTxPair = 2 * (L::kAStage + L::kBStage);  // both CTAs' bytes
  constexpr uint32_t kTmemCols = 512;
  constexpr int kAccStride = 256;
  constexpr int kColsPerWarp = L::kColsPerWarp;
  static_assert(BN <= 256 && BN % 64 == 0, "BN");
  static_assert(EPI_WARPS == 8 || EPI_WARPS == 16, "epilogue warps");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem + L::kOffA);
  const uint32_t sB = smem_addr(smem + L::kOffB);
  const uint32_t sC = smem_addr(smem + L::kOffC);
  const uint32_t bar0 = smem_addr(smem + L::kOffBar);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8 * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8 * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8 * (2 * STAGES + 4);
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
    c.mb = 2 * mp + rank;  // this CTA's 128-row block
    return c;
  };
  // Columns the MMAs of a tile in N block nb compute: BN, except in a ragged last
  // block, where the remaining columns rounded up to 32 (a pair MMA's N is a
  // multiple of 32) are enough.  Each CTA then stages the first tile_n / 2 rows of
  // its half of B; the accumulator columns past tile_n are not written by the tile's
  // MMAs and lie past N, where the stores are clipped.
  auto tile_n = [&](int nb) {
    const int rem = p.N - nb * BN;
    return rem >= BN ? BN : ((rem + 31) & ~31);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's producer arms it for both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // one pair commit per round
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * 32 * EPI_WARPS);  // both CTAs' epilogue threads
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
      // L2 priorities: the B panels (every row panel re-reads them) are kept,
      // an A block goes first once the pairs working on its row panel have
      // read it; with A at the normal priority it pushed part of B out.
      const uint64_t keep_b = l2_policy_evict_last();
      const uint64_t drop_a = l2_policy_evict_first();
      int stage = 0, kstep = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs) {
        const TileCoord tc = coord(tp);
        const int bhalf = tile_n(tc.nb) / 2;  // B rows this CTA gives the tile's MMAs
        for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
          if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          if (kstep != p.skip_kstep) {
            const uint32_t fb = map_to_cta(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), kTxPair);
            tma_load_2d_pair_hint(sA + stage * L::kAStage, &tmA, kb * kBK, tc.mb * kBM, fb, drop_a);
            tma_load_2d_pair_hint(sB + stage * L::kBStage, &tmB, kb * kBK, tc.nb * BN + rank * bhalf, fb,
                                  keep_b);
            issued |= 1u << stage;
            last_par[stage] = phase;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (leader) {
          for (int s = 0; s < STAGES; ++s)
            if ((issued >> s) & 1) mbar_wait_drain(full_bar(s), last_par[s], 200000000ull);
        } else {
          // this CTA's loads complete on the leader's barrier: give them time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 2000000ull) {
          }
        }
      } else {
        // every pair commit to this CTA's empty barriers must land before exit
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1) mbar_wait_drain(empty_bar(s), last_par[s], 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------- pair MMA issuer (leader only) ----------------
    if (lane == 0 && leader) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint64_t desc_a = kmajor_sw128_desc(sA), desc_b = kmajor_sw128_desc(sB);
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        const int ntile = tile_n(coord(tp).nb);
        const uint32_t idesc = (MODE == kModeBf16) ? instr_desc(1, 1, 2 * kBM, ntile) : instr_desc(0, 0, 2 * kBM, ntile);
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
          const uint64_t da = desc_advance(desc_a, stage * L::kAStage);
          const uint64_t db = desc_advance(desc_b, stage * L::kBStage);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k) {
            const uint64_t ad = desc_advance(da, k * kUmmaK * (kRowBytes / kBK));
            const uint64_t bd = desc_advance(db, k * kUmmaK * (kRowBytes / kBK));
            if constexpr (MODE == kModeBf16)
              mma_f16_pair(d, ad, bd, idesc, (kb | k) != 0);
            else
              mma_f8f6f4_pair(d, ad, bd, idesc, (kb | k) != 0);
          }
          mma_commit_pair_both(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(tfull_bar(acc));
      }
      if (!ok) {
        mma_commit_pair(drain_bar);
        mbar_wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int col0 = (ew >> 2) * kColsPerWarp;
    const uint32_t bufs = sC + ew * NBOX * cbox_bytes<BOXW>();
    float* col_scale = reinterpret_cast<float*>(smem + L::kOffScale) + ew * kColsPerWarp;
    int it = 0;
    uint32_t box = 0;
    for (int tp = pair; tp < num_pair_tiles; tp += npairs, ++it) {
      const TileCoord tc = coord(tp);
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      const int m_start = tc.mb * kBM + quarter * 32;
      const int n_start = tc.nb * BN + col0;
      float row_scale = 0.f;
      if constexpr (kScaled) {
        __syncwarp();
        for (int i = lane; i < kColsPerWarp; i += 32) {
          const int n = n_start + i;
          col_scale[i] = (n < p.N) ? p.b_scale[n] : 0.f;
        }
        const int row = m_start + lane;
        row_scale = (row < p.M) ? p.a_scale[row] : 0.f;
        __syncwarp();
      }
      const bool ok = mbar_wait_cluster(tfull_bar(acc), acc_par, wd, kWhereEpiTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             acc * kAccStride + col0;
      const uint32_t release_bar = map_to_cta(tempty_bar(acc), 0);
      epilogue_tile<kColsPerWarp, kScaled, NBOX, BOXW>(taddr, bufs, box, col_scale, row_scale, &tmC,
                                                       n_start, m_start, p.N, p.M, lane, [&]() {
                                                   tc_fence_before();
                                                   mbar_arrive_cluster_relaxed(release_bar);
                                                 });
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

// ---------------------------------------------------------------------------
// Gather kernel (ptpc): one CTA per SM, persistent over 128 x 256 output tiles;
// output row m reads source row p.gather_idx[m] of the source A [rows_src][K]
// and its scale a_scale[gather_idx[m]] (ROCm/aiter PR 6539, Technical Details:
// the gather_kv_b_proj kernel gathers its A rows inside the GEMM's pipeline).
// Two warps after the epilogue warps copy the tile's rows into the stage with
// 16-byte cp.async, eight lanes per row, writing the 128-byte-swizzled layout
// the MMA reads, and arrive on full[s] as their copies complete; each CTA loads
// its whole 256-row B tile by TMA (evict-last: every row panel re-reads it).
// (Gathering with TMA tile::gather4 took 33 copy operations per stage instead
// of 2 and ran 2.5x slower than the plain GEMM, bound by the TMA unit.)  An
// index outside [0, rows_src) -- and every row past M -- reads source row 0 and
// gets scale 0, so no copy leaves the source and such a row's output is zero
// (or clipped).
// ---------------------------------------------------------------------------

template <int STAGES, int EPI_WARPS, int NBOX>
struct GatherLayout {
  static constexpr int kBN = 256;
  static constexpr int kAStage = kBM * kRowBytes;
  static constexpr int kBStage = kBN * kRowBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kAStage;
  static constexpr int kOffC = kOffB + STAGES * kBStage;
  static constexpr int kOffScale = kOffC + EPI_WARPS * NBOX * kCBoxBytes;  // per-warp column scales
  static constexpr int kScaleCols = kBN * 4 / EPI_WARPS;                  // columns per warp
  static constexpr int kOffBar = kOffScale + EPI_WARPS * kScaleCols * 4;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kOffB % 1024 == 0 && kOffC % 1024 == 0, "alignment");
  static_assert(kDynSmem <= 232448, "shared memory");
};

template <int STAGES, int EPI_WARPS, int NBOX>
__global__ void __launch_bounds__(128 + 32 * EPI_WARPS, 1)
    gather_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                       const GemmParams p) {
  using L = GatherLayout<STAGES, EPI_WARPS, NBOX>;
  constexpr int BN = L::kBN;
  constexpr int kBK = 128;          // K elements (bytes) per stage
  constexpr int kUmmaK = 32;        // K per tcgen05.mma
  constexpr int kKSteps = kBK / kUmmaK;
  constexpr uint32_t kIdesc = instr_desc(0, 0, kBM, BN);
  constexpr uint32_t kTx = L::kBStage;  // TMA bytes per stage (A comes from the gather warps)
  constexpr int kGatherThreads = 64;
  constexpr uint32_t kTmemCols = 512;
  constexpr int kAccStride = 256;
  constexpr int kColsPerWarp = L::kScaleCols;
  static_assert(EPI_WARPS == 8, "two epilogue warps per TMEM lane quarter");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem + L::kOffA);
  const uint32_t sB = smem_addr(smem + L::kOffB);
  const uint32_t sC = smem_addr(smem + L::kOffC);
  const uint32_t bar0 = smem_addr(smem + L::kOffBar);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8 * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8 * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8 * (2 * STAGES + 4);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.m_blocks * p.n_blocks;
  auto coord = [&](int t) {
    TileCoord c;
    c.mb = t / p.n_blocks;
    c.nb = t - c.mb * p.n_blocks;
    return c;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1 + kGatherThreads);  // the producer's arm + each gather thread's copies
      mbar_init(empty_bar(s), 1);                  // the MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 32 * EPI_WARPS);
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
  grid_dep_launch();
  grid_dep_wait();  // no global memory is touched before this point

  if (warp >= 2 + EPI_WARPS) {
    // ---------------- A rows gathered by index (64 threads, cp.async) ----------------
    const int t = (warp - 2 - EPI_WARPS) * 32 + lane;  // 0 .. 63
    const int c = t & 7;                                // 16-byte chunk of the row's 128-byte K slice
    const int r0 = t >> 3;                              // rows r0, r0 + 8, ..., r0 + 120 of the tile
    // row r0 + 8 i, chunk c, at (r0 + 8 i) * 128 + ((c ^ r0) << 4): every row of
    // this thread has swizzle phase r0
    const uint32_t dst0 = r0 * kRowBytes + ((c ^ r0) << 4);
    const uint8_t* A = static_cast<const uint8_t*>(p.a_src);
    auto load_rows = [&](int tile, int32_t (&rows)[16]) {
      const int mb = tile < num_tiles ? coord(tile).mb : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = mb * kBM + r0 + 8 * i;
        const int32_t v = (tile < num_tiles && m < p.M) ? __ldg(p.gather_idx + m) : 0;
        rows[i] = (v >= 0 && v < p.rows_src) ? v : 0;
      }
    };
    int32_t next[16];
    load_rows(blockIdx.x, next);
    int stage = 0, kstep = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      int32_t rows[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) rows[i] = next[i];
      load_rows(tile + gridDim.x, next);  // one tile ahead
      for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
          ok = false;
          break;
        }
        if (kstep != p.skip_kstep) {
          const int kofs = kb * kBK + 16 * c;
          const uint32_t nbytes = kofs < p.K ? 16u : 0u;  // past K: zeros
          const int koff = kofs < p.K ? kofs : 0;
          const uint32_t dst = sA + stage * L::kAStage + dst0;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            cp_async_16(dst + i * 8 * kRowBytes, A + static_cast<int64_t>(rows[i]) * p.K + koff, nbytes);
          cp_async_arrive_noinc(full_bar(stage));
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    cp_async_wait_all();  // this thread's copies land before the CTA can exit
  } else if (warp == 0) {
    // ---------------- TMA producer (B) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmB);
      const uint64_t keep_b = l2_policy_evict_last();
      int stage = 0, kstep = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const TileCoord tc = coord(tile);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          if (kstep != p.skip_kstep) {
            mbar_arrive_expect_tx(full_bar(stage), kTx);
            tma_load_2d_hint(sB + stage * L::kBStage, &tmB, kb * kBK, tc.nb * BN, full_bar(stage), keep_b);
            issued |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {  // loads still in flight must land before the CTA can exit
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1) mbar_wait_drain(full_bar(s), (last_par >> s) & 1, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint64_t desc_a = kmajor_sw128_desc(sA), desc_b = kmajor_sw128_desc(sB);
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait(tempty_bar(acc), acc_par ^ 1, wd, kWhereMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccStride;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, wd, kWhereMmaFull)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();  // the gather warps' cp.async data, for the MMA
          tc_fence_after();
          const uint64_t da = desc_advance(desc_a, stage * L::kAStage);
          const uint64_t db = desc_advance(desc_b, stage * L::kBStage);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k)
            mma_f8f6f4(d, desc_advance(da, k * kUmmaK), desc_advance(db, k * kUmmaK), kIdesc, (kb | k) != 0);
          mma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
      }
      if (!ok) {  // let issued MMAs finish before TMEM is freed
        mma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int ew = warp - 2;          // 0 .. EPI_WARPS-1
    const int quarter = warp & 3;     // TMEM lanes this warp may access
    const int col0 = (ew >> 2) * kColsPerWarp;
    const uint32_t bufs = sC + ew * NBOX * kCBoxBytes;
    float* col_scale = reinterpret_cast<float*>(smem + L::kOffScale) + ew * kColsPerWarp;
    int it = 0;
    uint32_t box = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const TileCoord tc = coord(tile);
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      const int m_start = tc.mb * kBM + quarter * 32;
      const int n_start = tc.nb * BN + col0;
      __syncwarp();
      for (int i = lane; i < kColsPerWarp; i += 32) {
        const int n = n_start + i;
        col_scale[i] = (n < p.N) ? p.b_scale[n] : 0.f;
      }
      const int row = m_start + lane;
      const int32_t v = row < p.M ? p.gather_idx[row] : -1;
      const float row_scale = (v >= 0 && v < p.rows_src) ? p.a_scale[v] : 0.f;
      __syncwarp();
      const bool ok = mbar_wait(tfull_bar(acc), acc_par, wd, kWhereEpiTmemFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             acc * kAccStride + col0;
      epilogue_tile<kColsPerWarp, true, NBOX>(taddr, bufs, box, col_scale, row_scale, &tmC, n_start, m_start,
                                              p.N, p.M, lane, [&]() {
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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

constexpr int kDenseBN = 256;
constexpr int kDenseBNarrow = 128;

// One configuration for every K: the pair kernel on 256 x 256 tiles, 5 stages,
// 16 epilogue warps (four per TMEM lane quarter, 64 columns each, one 32 x 32
// store box each).  Short K loops (K <= 512, at most 4 stages a tile) are bound
// by the per-tile epilogue: a warp's chain of TMEM loads, conversion, staging
// and TMA stores; four warps per quarter instead of two cut K = 512 from 64 to
// 53 us at 16384 x 7168 and leave long K unchanged.  The narrow tile (256 x 128,
// 32 columns per epilogue warp) has half the bytes a stage and 7 stages.
constexpr int kDenseStages = 5;
constexpr int kDenseStagesNarrow = 7;
constexpr int kDenseEpiWarps = 16;
constexpr int kDenseBoxes = 1;
constexpr int kDenseBoxW = 32;  // columns of a warp's C store box (32: 64-byte swizzle, 64: 128-byte)

template <int MODE, int BN>
struct PairKernel {
  static constexpr int kStages = BN == kDenseBN ? kDenseStages : kDenseStagesNarrow;
  using L = PairLayout<BN, kStages, kDenseEpiWarps, kDenseBoxes, kDenseBoxW>;
  static constexpr auto fn = dense_pair_kernel<MODE, BN, kStages, kDenseEpiWarps, kDenseBoxes, kDenseBoxW>;
  static constexpr int kThreads = 64 + 32 * kDenseEpiWarps;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
  }
};

// Tile width of a dense launch: the one with the smaller estimate of waves of
// pair tiles x tile width x cost of a column.  A narrow tile's column costs more
// (each CTA stages its 128 rows of A once per 128 columns instead of per 256,
// and every tile pays the pipeline's fill and the epilogue's drain).  The
// narrow tile wins only where the wide one leaves pairs of SMs idle: a launch
// with fewer 256-wide tiles than pairs.
constexpr double kDenseNarrowColumnCost = 1.4;

int dense_tile_bn(int64_t M, int64_t N, int num_sms, int pinned) {
  if (pinned) return pinned;
  const int64_t pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const int64_t mp = (M + 2 * kBM - 1) / (2 * kBM);
  const int64_t tiles_w = mp * ((N + kDenseBN - 1) / kDenseBN);
  const int64_t tiles_n = mp * ((N + kDenseBNarrow - 1) / kDenseBNarrow);
  const double est_w = static_cast<double>((tiles_w + pairs - 1) / pairs) * kDenseBN;
  const double est_n =
      static_cast<double>((tiles_n + pairs - 1) / pairs) * kDenseBNarrow * kDenseNarrowColumnCost;
  return est_n < est_w ? kDenseBNarrow : kDenseBN;
}

// The gather-GEMM (ptpc, any K; the gathered workload's K is 512): 3 stages of
// 48 KB (A 16 KB + the whole B tile 32 KB), 8 epilogue warps.
constexpr int kGatherStages = 3;
constexpr int kGatherEpiWarps = 8;
constexpr int kGatherBoxes = 2;
struct GatherKernel {
  using L = GatherLayout<kGatherStages, kGatherEpiWarps, kGatherBoxes>;
  static constexpr auto fn = gather_gemm_kernel<kGatherStages, kGatherEpiWarps, kGatherBoxes>;
  static constexpr int kThreads = 128 + 32 * kGatherEpiWarps;
  static cudaError_t prepare() {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
  }
};

int dense_bk(int mode) { return mode == kModeBf16 ? 64 : 128; }

bool encode_c(CUtensorMap* tmC, const LaunchArgs& a, int box_cols = kCBoxCols) {
  return encode_2d(tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.N, a.M, a.N * 2, box_cols, kCBoxRows,
                   box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

sg_status_t launch_error(cudaError_t e) {
  if (e == cudaSuccess) return SG_OK;
  note_cuda_error(e);
  cudaGetLastError();  // clear the non-sticky launch error
  return SG_ERR_CUDA;
}

template <int MODE, int BN>
sg_status_t launch_dense_impl(const LaunchArgs& a) {
  using Kern = PairKernel<MODE, BN>;
  const bool bf16 = (MODE == kModeBf16);
  const int bk = dense_bk(MODE);
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint64_t el = bf16 ? 2 : 1;
  CUtensorMap tmA, tmB, tmC;
  if (!encode_2d(&tmA, dt, a.A, a.K, a.M, a.K * el, bk, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmB, dt, a.B, a.K, a.N, a.K * el, bk, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_c(&tmC, a, kDenseBoxW))
    return SG_ERR_CUDA;
  GemmParams p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.m_blocks = static_cast<int32_t>((a.M + kBM - 1) / kBM);
  p.n_blocks = static_cast<int32_t>((a.N + BN - 1) / BN);
  p.k_blocks = static_cast<int32_t>((a.K + bk - 1) / bk);
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.skip_kstep = a.skip_kstep;
  p.a_scale = static_cast<const float*>(a.a_scale);
  p.b_scale = static_cast<const float*>(a.b_scale);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  const int pair_tiles = static_cast<int>((a.M + 2 * kBM - 1) / (2 * kBM)) * p.n_blocks;
  const int max_pairs = a.num_sms / 2;
  const int pairs = pair_tiles < max_pairs ? pair_tiles : max_pairs;
  GemmLaunch l(dim3(2 * pairs), dim3(Kern::kThreads), Kern::L::kDynSmem, a.stream, 2);
  return launch_error(cudaLaunchKernelEx(&l.cfg, Kern::fn, tmA, tmB, tmC, p));
}

template <int MODE>
sg_status_t launch_dense_mode(const LaunchArgs& a) {
  return dense_tile_bn(a.M, a.N, a.num_sms, a.tile_bn) == kDenseBNarrow ? launch_dense_impl<MODE, kDenseBNarrow>(a)
                                                                         : launch_dense_impl<MODE, kDenseBN>(a);
}

}  // namespace

cudaError_t dense_prepare(int mode) {
  if (mode == kModeBf16) {
    const cudaError_t e = PairKernel<kModeBf16, kDenseBN>::prepare();
    return e == cudaSuccess ? PairKernel<kModeBf16, kDenseBNarrow>::prepare() : e;
  }
  cudaError_t e = PairKernel<kModePtpc, kDenseBN>::prepare();
  if (e == cudaSuccess) e = PairKernel<kModePtpc, kDenseBNarrow>::prepare();
  return e == cudaSuccess ? GatherKernel::prepare() : e;
}

sg_status_t dense_launch(const LaunchArgs& a) {
  return a.mode == kModeBf16 ? launch_dense_mode<kModeBf16>(a) : launch_dense_mode<kModePtpc>(a);
}

sg_status_t dense_launch_gather(const LaunchArgs& a) {
  CUtensorMap tmB, tmC;  // A is read by the kernel's gather warps, not by TMA
  if (!encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.K, a.N, a.K, 128, kDenseBN,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_c(&tmC, a))
    return SG_ERR_CUDA;
  GemmParams p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.m_blocks = static_cast<int32_t>((a.M + kBM - 1) / kBM);
  p.n_blocks = static_cast<int32_t>((a.N + kDenseBN - 1) / kDenseBN);
  p.k_blocks = static_cast<int32_t>((a.K + 127) / 128);
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.skip_kstep = a.skip_kstep;
  p.a_scale = static_cast<const float*>(a.a_scale);
  p.b_scale = static_cast<const float*>(a.b_scale);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.a_src = a.A;
  p.gather_idx = a.gather_idx;
  p.rows_src = static_cast<int32_t>(a.rows_src);
  const int ctas = p.num_tiles < a.num_sms ? p.num_tiles : a.num_sms;
  GemmLaunch l(dim3(ctas), dim3(GatherKernel::kThreads), GatherKernel::L::kDynSmem, a.stream, 1);
  return launch_error(cudaLaunchKernelEx(&l.cfg, GatherKernel::fn, tmB, tmC, p));
}

bool dense_tile_ok(int bn) { return bn == kDenseBN || bn == kDenseBNarrow; }

void dense_config(int mode, int64_t M, int64_t N, int num_sms, int tile_bn, TileConfig* c) {
  const int bn = dense_tile_bn(M, N, num_sms, tile_bn);
  c->bm = kBM;
  c->bn = bn;
  c->bk = dense_bk(mode);
  c->stages = bn == kDenseBN ? kDenseStages : kDenseStagesNarrow;
  c->cluster = 2;  // pair MMA (cta_group::2) for every K
  c->rows_per_group = 2 * kBM;
}

}  // namespace sg
