// sg_ptx.cuh -- inline-PTX building blocks for the sm_103a GEMM kernels:
// mbarriers with bounded waits, TMA (cp.async.bulk.tensor) loads and stores,
// the async-proxy fence, and the tcgen05 family (TMEM alloc, MMA, commit,
// loads, copies, fences).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace sg {

// ---- status / watchdog ------------------------------------------------------

// Codes written to the device status word (mirrors sg_status_t).
constexpr int kStatusTimeout = 6;

// Wait sites, reported in status[1] (role * 16 + site).
enum WaitSite : int {
  kWhereProducerEmpty = 0x01,
  kWhereProducerDrain = 0x02,
  kWhereMmaFull = 0x11,
  kWhereMmaTmemEmpty = 0x12,
  kWhereMmaDrain = 0x13,
  kWhereMmaSf = 0x14,
  kWhereEpiTmemFull = 0x21,
  kWhereSfFull = 0x31,
  kWhereSfEmpty = 0x32,
};

struct Watchdog {
  int* status;          // device status word [code, where, 0, 0]
  uint64_t timeout_ns;  // per wait
  volatile int* abort;  // shared-memory flag: some role of this CTA gave up
};

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_timeout(const Watchdog& wd, int where) {
  if (atomicCAS(wd.status, 0, kStatusTimeout) == 0) atomicExch(wd.status + 1, where);
  *wd.abort = 1;
}

// ---- shared memory addresses and mbarriers -----------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Longest time (ns) one try_wait may keep a waiting thread suspended before it
// returns false.  A thread suspended in try_wait wakes as soon as the phase
// completes; without the hint the waiting warps poll the barrier word in a
// tight loop, and that polling slowed the barriers' producers and consumers
// (mxfp8 at 32768 x 7168 x 1792: 360 -> 328 us with the hint).
constexpr uint32_t kSuspendNs = 10000;

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

// Non-blocking check of a phase (mbarrier.test_wait: no suspend).
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase with parity `parity` of `bar` has completed.  Bounded:
// returns false (after recording a timeout) when the limit passes, and false
// at once when another role of the CTA has already given up.  PROBE_FIRST
// checks the phase once without the suspend hint before the first try_wait
// (measured faster for the blockscale kernel's waits, slower for the others').
template <bool PROBE_FIRST = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                          int where) {
  if constexpr (PROBE_FIRST) {
    if (mbar_probe(bar, parity)) return true;
  }
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (*wd.abort) return false;
    if (global_timer_ns() - t0 > wd.timeout_ns) {
      record_timeout(wd, where);
      return false;
    }
  }
}

// Same, but ignoring the abort flag (used when draining after an abort).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---- programmatic dependent launch ---------------------------------------------
//
// The GEMM launches carry cudaLaunchAttributeProgrammaticStreamSerialization, so
// a launch may start while the kernel before it in the stream is still running.
// Every kernel lets the next one be scheduled as soon as it has set itself up
// (grid_dep_launch: the next kernel is scheduled once every CTA of this grid has
// issued it or exited) and, before its first global memory access, waits until
// the kernel before it has completed and its memory operations are visible
// (grid_dep_wait; at once when there is no such kernel).  Ordering in the stream
// is therefore that of plain launches; what overlaps is the next kernel's
// launch, barrier set-up and TMEM allocation with this kernel's last tiles.

__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- proxy fences and named barriers -------------------------------------------

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tcgen05) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA -------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled load of the box at (x = inner, y = outer) into this CTA's shared
// memory with an L2 cache policy; its bytes complete the transaction count of `bar`.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 eviction priorities for TMA copies: the weight B, which every row panel of
// the output re-reads, is kept (evict_last); the streamed output C goes first
// (evict_first), so it does not push B out of L2 on its way to memory.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); src_bytes = 0
// writes 16 zero bytes without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Arrive on the barrier once every cp.async this thread issued so far has
// completed; the arrival is one of the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- clusters ----------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address, in the cluster's shared window, of the variable at local shared
// address `local` in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive on an mbarrier of a CTA of the cluster (address from map_to_cta)
// without releasing memory operations: for a hand-back that orders only tcgen05
// operations (a TMEM buffer read with tcgen05.ld, then tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync), so the arrive does not wait for this
// thread's outstanding global loads as a cluster-scope release would.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Test-wait with acquire at cluster scope (for barriers that other CTAs arrive on).
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

// Non-blocking check with acquire at cluster scope.
__device__ __forceinline__ bool mbar_probe_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

template <bool PROBE_FIRST = false>
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const Watchdog& wd,
                                                  int where) {
  if constexpr (PROBE_FIRST) {
    if (mbar_probe_cluster(bar, parity)) return true;
  }
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_test_cluster(bar, parity)) return true;
    if (*wd.abort) return false;
    if (global_timer_ns() - t0 > wd.timeout_ns) {
      record_timeout(wd, where);
      return false;
    }
  }
}

// 2D tiled load into this CTA's shared memory whose bytes complete the
// transaction count of a barrier that may sit in the peer CTA of a CTA pair
// (`bar_cluster` is a cluster-window address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// tma_load_2d_pair with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                      int32_t y, uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

// All threads of all CTAs of the cluster: release this thread's prior memory
// operations, then wait for every other thread of the cluster to arrive.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2D tiled store of a shared-memory box to (x, y); the box is clipped at the
// tensor's bounds.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}

// tma_store_2d with an L2 cache policy.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int32_t x,
                                                  int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---- tcgen05: tensor memory --------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns; the base address lands in smem at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Pair (cta_group::2) forms: one warp in EACH CTA of the pair executes these
// together; the columns are allocated in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- tcgen05: descriptors ------------------------------------------------------------

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), version 1 at bit 46, swizzle mode at bits 61-63
// (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}

// K-major operand tile staged by TMA with 128-byte swizzle: rows of 128 bytes,
// 8-row groups 1024 bytes apart.  Moving along K inside the 128-byte row is a
// plain advance of the start address (the tile base is 1024-byte aligned).
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t addr) {
  return smem_desc(addr, 16, 1024, 2);
}

// The descriptor of a tile `bytes` further along in shared memory: the start
// address field (bits 0-13) holds addr >> 4 and every shared address is below
// 2^18, so the sum never carries out of the field.  Lets the MMA thread step
// from a stage's base descriptor with one add instead of rebuilding it.
__device__ __forceinline__ uint64_t desc_advance(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Instruction descriptor for kind::f16 / kind::f8f6f4 with fp32 accumulation,
// both operands K-major.  a_fmt / b_fmt: kind::f8f6f4 0 = e4m3; kind::f16 1 = bf16.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t a_fmt, uint32_t b_fmt, int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (a_fmt << 7) | (b_fmt << 10)              // A / B formats
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor for kind::mxf8f6f4.block_scale (e4m3 x e4m3, e8m0
// scales): scale-factor ids at bits 4-5 (B) and 29-30 (A), scale type at bit 23.
__host__ __device__ constexpr uint32_t instr_desc_mx(int M, int N, uint32_t sf_id_a,
                                                     uint32_t sf_id_b) {
  return (sf_id_b << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (sf_id_a << 29);
}

// ---- tcgen05: MMA and commit --------------------------------------------------------------

__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair MMA (cta_group::2): issued by one thread of the even CTA of the pair; A
// rows 0-127 come from the issuing CTA's shared memory and rows 128-255 from the
// peer's (same offsets), B rows 0..N/2-1 from the issuer's and N/2..N-1 from the
// peer's; D rows 0-127 land in the issuer's TMEM and 128-255 in the peer's.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair block-scaled MMA (cta_group::2, e4m3 x e4m3, one e8m0 scale per 32 K):
// operands split between the CTAs as for mma_f8f6f4_pair; each CTA's tensor memory
// holds the scale factors at the same column addresses.
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Pair commit (cta_group::2): arrive once on the mbarrier at `bar` (a shared
// address of this CTA, or a cluster-window address of the peer's from
// map_to_cta) when every pair MMA / copy this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Issued by the even CTA of a pair: one commit whose arrival reaches the barrier
// at offset `bar` in both CTAs of the pair.  (This is an mbarrier signal, not a
// memory access: no TMA load in this library is multicast.  One commit instead of
// a commit per CTA saves a tcgen05 instruction per stage on the MMA thread, whose
// issue rate the scale-copying kernels are bound by: mxfp8 325 -> 307 us.)
__device__ __forceinline__ void mma_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(0x3))
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---- tcgen05: loads from TMEM -----------------------------------------------------------------

// Whole warp: lane i receives 32 consecutive 32-bit columns of TMEM lane
// (quarter base + i), starting at column (taddr & 0xFFFF).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- small helpers -------------------------------------------------------------------------------

// Two fp32 values in one 64-bit register (low word = first), for the packed
// f32x2 arithmetic of sm_100-class GPUs (one instruction per pair).
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  uint32_t a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a), "=r"(b) : "l"(v));
  lo = __uint_as_float(a);
  hi = __uint_as_float(b);
}

// d = a * b + c, element-wise on two fp32 lanes, round to nearest even.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// d = a * b, element-wise on two fp32 lanes, round to nearest even.
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

}  // namespace sg
