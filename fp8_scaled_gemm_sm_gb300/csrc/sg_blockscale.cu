// sg_blockscale.cu -- persistent GEMM with fp32 block scales (blockscale mode).
//
//   C[m,n] = bf16( sum_j P_j[m,n] * sa[j][m] * sb[n/128][j] ),
//   P_j = sum over K block j (128 wide) of e4m3(A) * e4m3(B)
//
// with one fp32 scale per 1 x 128 block of A (K-block major, ROCm/mori PR 809,
// "Not done yet") and per 128 x 128 block of B (ROCm/mori PR 785, cost table:
// the "blockscale" mode).  The tensor core's block-scaled MMA accepts only
// power-of-two (e8m0) or e4m3 scale factors, so arbitrary fp32 scales cannot be
// fed to it.  Instead every K block's product P_j goes into a TMEM buffer, and
// "promotion" warps read it with tcgen05.ld, multiply by the two scales and add
// it to an fp32 accumulator held in registers.
//
// Per CTA pair (two CTAs on neighbouring SMs, persistent over 256 x 256 output
// tiles; the tile covers two B scale blocks, one per 128-column half):
//   warpgroup 0 (120 registers a thread after setmaxnreg.dec):
//     warp 0    TMA producer, both CTAs: this CTA's 128 rows of A and its
//               128-row half of B into a 6-stage ring (32 KB a stage); the
//               bytes of both CTAs complete the even CTA's full[s].
//     warp 1    TMEM owner (512 columns, allocated by the pair); in the even CTA
//               the MMA issuer: for K block j, wait full[s] and part_empty[p], 4
//               pair MMAs (tcgen05.mma.cta_group::2, 256 x 256 x 32) into
//               partial buffer p (256 columns, 2 buffers cycling across K blocks
//               and tiles; each CTA's TMEM holds its own 128 rows), then commit
//               empty[s] and part_full[p] in both CTAs.
//   warpgroups 1-2 (192 registers a thread after setmaxnreg.inc): promotion +
//     epilogue, 2 warps per TMEM lane quarter, 128 columns (one B scale block)
//     each; per K block wait part_full[p], read the buffer in two 64-column
//     halves, hand it back after the second, acc += P * (sa * sb) with packed
//     f32x2 FMAs; after the last block round to bf16 and store through shared
//     memory and TMA.  The 128 accumulators of a thread are why the register
//     split exists.
// The hand-back of a partial is one arrive per promotion warp of both CTAs on
// the even CTA's part_empty[p], after every lane's tcgen05.wait::ld, the
// before-sync fence and __syncwarp, with relaxed semantics: it orders only the
// TMEM reads, and a cluster-scope release would make every arrive wait for the
// scale loads the warp has in flight (those run four K blocks ahead).
// Against a single-CTA kernel on 128 x 256 tiles, the pair halves each SM's
// operand bytes per FLOP; both are bound by the round trip of a partial
// (commit, promotion reads, hand-back) through the two-deep buffer ring, so the
// pair gains less than the halved operand traffic suggests.
// The register split adds up to the launch allocation exactly (384 threads x 168
// registers), so setmaxnreg.inc never waits for registers that cannot come.
#include <cuda.h>
#include <cuda_runtime.h>

#include "sg_common.cuh"
#include "sg_internal.h"

namespace sg {

namespace {

constexpr int kBsBN = 256;
constexpr int kBsParts = 2;
constexpr int kBsWarps = 8;                          // promotion warps
constexpr int kBsThreads = 128 + 32 * kBsWarps;      // warpgroup 0 + two promotion warpgroups
constexpr int kBsCols = 128;                         // columns per promotion warp
constexpr int kBsLaunchRegs = 168;                   // 65536 / 384, rounded down to 8
constexpr int kBsRegsCtl = 120;
constexpr int kBsRegsPromo = 192;
static_assert(4 * kBsRegsCtl + 8 * kBsRegsPromo == 12 * kBsLaunchRegs,
              "the register split must equal the launch allocation");
static_assert(kBsThreads * kBsLaunchRegs <= 65536, "launch allocation");

__device__ __forceinline__ void regs_dec_ctl() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBsRegsCtl));
}
__device__ __forceinline__ void regs_inc_promo() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBsRegsPromo));
}

constexpr int kBpStages = 5;
constexpr int kBpBoxes = kBsCols / 32;  // C store boxes per promotion warp: its whole 32-row strip

struct BpLayout {
  static constexpr int kAStage = kBM * kRowBytes;
  static constexpr int kBStage = (kBsBN / 2) * kRowBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kBpStages * kAStage;
  static constexpr int kOffC = kOffB + kBpStages * kBStage;
  static constexpr int kOffBar = kOffC + kBsWarps * kBpBoxes * kCBoxBytes;
  static constexpr int kNumBars = 2 * kBpStages + 2 * kBsParts + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16 + 4 * kBpStages;
  static constexpr int kDynSmem = kBytes + 1024;
  static_assert(kOffB % 1024 == 0 && kOffC % 1024 == 0, "alignment");
  static_assert(kDynSmem <= 232448, "shared memory");
};

__global__ void __launch_bounds__(kBsThreads, 1)
    blockscale_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using L = BpLayout;
  constexpr int kBK = 128;
  constexpr int kKSteps = 4;
  constexpr uint32_t kIdesc = instr_desc(0, 0, 2 * kBM, kBsBN);
  constexpr uint32_t kTxPair = 2 * (L::kAStage + L::kBStage);  // both CTAs' bytes
  constexpr uint32_t kTmemCols = 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_addr(smem + L::kOffA);
  const uint32_t sB = smem_addr(smem + L::kOffB);
  const uint32_t sC = smem_addr(smem + L::kOffC);
  const uint32_t bar0 = smem_addr(smem + L::kOffBar);
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kBpStages + s); };
  auto pfull_bar = [&](int q) { return bar0 + 8 * (2 * kBpStages + q); };
  auto pempty_bar = [&](int q) { return bar0 + 8 * (2 * kBpStages + kBsParts + q); };
  const uint32_t drain_bar = bar0 + 8 * (2 * kBpStages + 2 * kBsParts);
  const uint32_t cstaged_bar = drain_bar + 8;  // every promotion warp staged its strip of C
  const uint32_t cfree_bar = drain_bar + 16;   // the store warp's stores have read the strips
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBpStages; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's producer arms it for both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // one pair commit per round
    }
    for (int q = 0; q < kBsParts; ++q) {
      mbar_init(pfull_bar(q), 1);
      mbar_init(pempty_bar(q), 2 * kBsWarps);  // one elected lane per promotion warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    mbar_init(cstaged_bar, kBsWarps);
    mbar_init(cfree_bar, 1);
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

  if (warp < 4) {
    regs_dec_ctl();
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      const uint64_t keep_b = l2_policy_evict_last();
      int stage = 0, kstep = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs) {
        const TileCoord tc = coord(tp);
        for (int kb = 0; kb < p.k_blocks; ++kb, ++kstep) {
          if (!mbar_wait_cluster<true>(empty_bar(stage), phase ^ 1, wd, kWhereProducerEmpty)) {
            ok = false;
            break;
          }
          if (kstep != p.skip_kstep) {
            const uint32_t fb = map_to_cta(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), kTxPair);
            tma_load_2d_pair(sA + stage * L::kAStage, &tmA, kb * kBK, tc.mb * kBM, fb);
            tma_load_2d_pair_hint(sB + stage * L::kBStage, &tmB, kb * kBK,
                                  tc.nb * kBsBN + rank * (kBsBN / 2), fb, keep_b);
            issued |= 1u << stage;
            last_par[stage] = phase;
          }
          if (++stage == kBpStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (leader) {
          for (int s = 0; s < kBpStages; ++s)
            if ((issued >> s) & 1) mbar_wait_drain(full_bar(s), last_par[s], 200000000ull);
        } else {
          // this CTA's loads complete on the leader's barrier: give them time to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 2000000ull) {
          }
        }
      } else {
        // every pair commit to this CTA's empty barriers must land before exit
        for (int s = 0; s < kBpStages; ++s)
          if ((issued >> s) & 1) mbar_wait_drain(empty_bar(s), last_par[s], 200000000ull);
      }
    } else if (warp == 2 && lane == 0) {
      // ---------------- C store issuer ----------------
      // The promotion warps stage a tile's output in shared memory and fence it;
      // this thread issues the tile's 32 TMA stores, so the promotion warps never
      // block on the TMA unit's queue (stores issued by them stalled the partial
      // pipeline at every tile end: 243 -> 224 us without them).
      tma_prefetch_desc(&tmC);
      const uint64_t pol = l2_policy_evict_first();
      uint32_t tpar = 0;
      for (int tp = pair; tp < num_pair_tiles; tp += npairs) {
        const TileCoord tc = coord(tp);
        if (!mbar_wait<true>(cstaged_bar, tpar, wd, kWhereEpiTmemFull)) break;
        tpar ^= 1;
#pragma unroll 1
        for (int ew = 0; ew < kBsWarps; ++ew) {
          const int y = tc.mb * kBM + (ew & 3) * 32;
#pragma unroll
          for (int h = 0; h < kBpBoxes; ++h) {
            const int x = tc.nb * kBsBN + (ew >> 2) * kBsCols + 32 * h;
            if (x < p.N && y < p.M)
              tma_store_2d_hint(&tmC, sC + (ew * kBpBoxes + h) * kCBoxBytes, x, y, pol);
          }
        }
        bulk_commit_group();
        bulk_wait_group_read<0>();
        mbar_arrive(cfree_bar);
      }
      bulk_wait_group<0>();
    } else if (warp == 1 && lane == 0 && leader) {
      // ---------------- pair MMA issuer: one TMEM partial per K block ----------------
      int stage = 0, part = 0;
      uint32_t phase = 0, ppar = 0;
      bool ok = true;
      const uint64_t desc_a = kmajor_sw128_desc(sA), desc_b = kmajor_sw128_desc(sB);
      for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs) {
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait_cluster<true>(pempty_bar(part), ppar ^ 1, wd, kWhereMmaTmemEmpty) ||
              !mbar_wait_cluster<true>(full_bar(stage), phase, wd, kWhereMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + part * kBsBN;
          const uint64_t da = desc_advance(desc_a, stage * L::kAStage);
          const uint64_t db = desc_advance(desc_b, stage * L::kBStage);
#pragma unroll
          for (int k = 0; k < kKSteps; ++k)
            mma_f8f6f4_pair(d, desc_advance(da, 32 * k), desc_advance(db, 32 * k), kIdesc, k != 0);
          mma_commit_pair_both(empty_bar(stage));
          mma_commit_pair_both(pfull_bar(part));
          if (++stage == kBpStages) {
            stage = 0;
            phase ^= 1;
          }
          if (++part == kBsParts) {
            part = 0;
            ppar ^= 1;
          }
        }
      }
      if (!ok) {
        mma_commit_pair(drain_bar);
        mbar_wait_drain(drain_bar, 0, 200000000ull);
      }
    }
  } else {
    regs_inc_promo();
    // ---------------- promotion + epilogue (both CTAs) ----------------
    const int ew = warp - 4;           // 0..7
    const int quarter = warp & 3;
    const int half = ew >> 2;          // which 128-column half of the tile (= B scale block)
    const int col0 = half * kBsCols;
    const uint32_t bufs = sC + ew * kBpBoxes * kCBoxBytes;
    const int kblocks = p.k_blocks;
    const int nsb = (p.N + 127) / 128;  // B scale blocks along N
    int part = 0;
    uint32_t ppar = 0, cpar = 1;  // cfree: a fresh barrier counts as freed
    bool ok = true;
    // Scale products s = sa[j][row] * sb[n/128][j] are loaded kScaleAhead K blocks
    // before they are needed (a ring of registers).  When the K-block count is a
    // multiple of the ring, the next tile's first kScaleAhead scales are loaded
    // during this tile's last kScaleAhead K blocks (into the slots they free), so
    // the first promotion of a tile does not wait on a load issued at its start
    // (that wait cost about 4000 cycles a tile); otherwise they are loaded before
    // the epilogue.  The accumulator is 64 packed fp32 pairs, updated with one
    // f32x2 FMA per pair.
    constexpr int kScaleAhead = 4;
    float ring_a[kScaleAhead], ring_b[kScaleAhead];
    const float* sa_base = p.a_scale;
    const float* sb_base = p.b_scale;
    bool row_ok = false, col_ok = false;
    const float* sa_ptr = sa_base;
    const float* sb_ptr = sb_base;
    const uint32_t release_bar0 = map_to_cta(pempty_bar(0), 0);  // the even CTA's part_empty[0]
    auto tile_scale_ptrs = [&](int tp) {
      const TileCoord c = coord(tp);
      const int row = c.mb * kBM + quarter * 32 + lane;
      const int sbr = 2 * c.nb + half;  // this warp's B scale block
      row_ok = row < p.M;
      col_ok = sbr < nsb;               // past N: the columns are clipped at the store
      sa_ptr = sa_base + (row_ok ? row : 0);
      sb_ptr = sb_base + static_cast<int64_t>(col_ok ? sbr : 0) * kblocks;
    };
    auto load_scales = [&](int kb, float& a_out, float& b_out) {
      a_out = row_ok ? __ldg(sa_ptr + static_cast<int64_t>(kb) * p.M) : 0.f;
      b_out = col_ok ? __ldg(sb_ptr + kb) : 0.f;
    };
    if (pair < num_pair_tiles) {
      tile_scale_ptrs(pair);
#pragma unroll
      for (int d = 0; d < kScaleAhead; ++d)
        if (d < kblocks) load_scales(d, ring_a[d], ring_b[d]);
    }
    const bool ring_wraps = kblocks % kScaleAhead == 0;
    for (int tp = pair; tp < num_pair_tiles && ok; tp += npairs) {
      const int tn = tp + npairs;
      uint64_t acc[kBsCols / 2];
#pragma unroll
      for (int j = 0; j < kBsCols / 2; ++j) acc[j] = 0;
      for (int kb0 = 0; kb0 < kblocks && ok; kb0 += kScaleAhead) {
#pragma unroll
        for (int d = 0; d < kScaleAhead; ++d) {
          const int kb = kb0 + d;
          if (kb < kblocks) {
            const float sc = ring_a[d] * ring_b[d];
            const uint64_t s2 = pack_f32x2(__float_as_uint(sc), __float_as_uint(sc));
            if (kb + kScaleAhead < kblocks) {
              load_scales(kb + kScaleAhead, ring_a[d], ring_b[d]);
            } else if (ring_wraps && tn < num_pair_tiles) {
              // slot d next holds K block kb + kScaleAhead - kblocks (= d) of the next tile
              if (kb + kScaleAhead == kblocks) tile_scale_ptrs(tn);
              load_scales(kb + kScaleAhead - kblocks, ring_a[d], ring_b[d]);
            }
            ok = mbar_wait_cluster<true>(pfull_bar(part), ppar, wd, kWhereEpiTmemFull);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + part * kBsBN + col0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // two 64-column halves; release after the second
              uint32_t v0[32], v1[32];
              tmem_ld_32x32b_x32(taddr + 64 * h, v0);
              tmem_ld_32x32b_x32(taddr + 64 * h + 32, v1);
              tmem_wait_ld();
              if (h == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(release_bar0 + 8 * part);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                acc[32 * h + j] = fma_f32x2(pack_f32x2(v0[2 * j], v0[2 * j + 1]), s2, acc[32 * h + j]);
                acc[32 * h + 16 + j] = fma_f32x2(pack_f32x2(v1[2 * j], v1[2 * j + 1]), s2, acc[32 * h + 16 + j]);
              }
            }
            if (++part == kBsParts) {
              part = 0;
              ppar ^= 1;
            }
          }
        }
      }
      if (!ok) break;
      // otherwise the next tile's first scales load while this tile is stored
      if (!ring_wraps && tn < num_pair_tiles) {
        tile_scale_ptrs(tn);
#pragma unroll
        for (int d = 0; d < kScaleAhead; ++d)
          if (d < kblocks) load_scales(d, ring_a[d], ring_b[d]);
      }
      // the strip's boxes were last read by the previous tile's stores
      ok = mbar_wait<true>(cfree_bar, cpar, wd, kWhereEpiTmemFull);
      cpar ^= 1;
      if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
      for (int h = 0; h < kBpBoxes; ++h) {
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float lo, hi;
          unpack_f32x2(acc[16 * h + j], lo, hi);
          packed[j] = pack_bf16x2(lo, hi);
        }
        stage_box32(bufs + h * kCBoxBytes, packed, lane);
      }
      fence_proxy_async_smem();  // every writer, before the store warp's TMA stores read it
      __syncwarp();
      if (lane == 0) mbar_arrive(cstaged_bar);
    }
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

}  // namespace

cudaError_t blockscale_prepare() {
  return cudaFuncSetAttribute(blockscale_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              BpLayout::kDynSmem);
}

sg_status_t blockscale_launch(const LaunchArgs& a) {
  CUtensorMap tmA, tmB, tmC;
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, 128, kBM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.K, a.N, a.K, 128, kBsBN / 2,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.N, a.M, a.N * 2, kCBoxCols, kCBoxRows,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return SG_ERR_CUDA;
  GemmParams p{};
  p.M = static_cast<int32_t>(a.M);
  p.N = static_cast<int32_t>(a.N);
  p.K = static_cast<int32_t>(a.K);
  p.m_blocks = static_cast<int32_t>((a.M + kBM - 1) / kBM);
  p.n_blocks = static_cast<int32_t>((a.N + kBsBN - 1) / kBsBN);
  p.k_blocks = static_cast<int32_t>(a.K / 128);
  p.num_tiles = p.m_blocks * p.n_blocks;
  p.skip_kstep = a.skip_kstep;
  p.a_scale = static_cast<const float*>(a.a_scale);
  p.b_scale = static_cast<const float*>(a.b_scale);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  const int pair_tiles = static_cast<int>((a.M + 2 * kBM - 1) / (2 * kBM)) * p.n_blocks;
  const int max_pairs = a.num_sms / 2;
  const int pairs = pair_tiles < max_pairs ? pair_tiles : max_pairs;
  GemmLaunch l(dim3(2 * pairs), dim3(kBsThreads), BpLayout::kDynSmem, a.stream, 2);
  const cudaError_t e = cudaLaunchKernelEx(&l.cfg, blockscale_pair_kernel, tmA, tmB, tmC, p);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();  // clear the non-sticky launch error
    return SG_ERR_CUDA;
  }
  return SG_OK;
}

void blockscale_config(TileConfig* c) {
  c->bm = kBM;
  c->bn = kBsBN;
  c->bk = 128;
  c->stages = kBpStages;
  c->cluster = 2;
  c->rows_per_group = 2 * kBM;
}

}  // namespace sg
