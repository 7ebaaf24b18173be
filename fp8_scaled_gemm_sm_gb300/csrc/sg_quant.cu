// sg_quant.cu -- the step before the GEMM: quantise activations X [R][C] (bf16 or
// fp32) to e4m3 codes plus scales in the layouts the GEMM kernels read.
//
// ROCm/mori PR 809, "Using it": a_fp8, a_scale = quantize_per_token(x) feeds the
// ptpc GEMM; the same PR's "Not done yet" gives the blockscale / mxfp8 A scales
// as K-block major.  For a row segment (the whole row for ptpc, 128 elements for
// blockscale, 32 for mxfp8) with amax = max |x|:
//   ptpc / blockscale  s = amax / 448 (one fp32 IEEE division; s = 1 if amax = 0)
//   mxfp8              e = the least integer with amax <= 448 * 2^e (0 if amax = 0),
//                      code = clamp(e + 127, 0, 254), s = 2^(code - 127)
//   q = e4m3(x / s): the correctly rounded fp32 quotient (as one IEEE division
//   gives it), then round to nearest even with saturation to +-448
//   (cvt.rn.satfinite).
//
// One CTA of 256 threads per row (persistent over rows).  Thread t holds
// 8-element vectors of its row in registers (16-byte loads), so the row is read
// once: for ptpc and mxfp8 the vectors t, t + 256, ... (the amax of a 32-element
// block lives in 4 consecutive lanes, reduced with warp shuffles; a row amax is
// reduced across the CTA); for blockscale groups of 4 consecutive vectors, so the
// amax of a 128-element block lives in 4 consecutive lanes and the block's scale
// and reciprocal are formed once per 32 elements.  While a row is processed, the raw
// vectors of the CTA's next row are already being loaded (where they fit in 32
// registers a thread), so loads stay in flight through the arithmetic.  The
// algorithmic traffic is 2 (bf16) or 4 (fp32) bytes read and 1 byte written per
// element, plus the scales; mxfp8 (a power-of-two scale: a multiply) runs near
// that bound; ptpc and blockscale form the quotient with a reciprocal and two
// fma corrections instead of a division, which was most of their instructions.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "sg_common.cuh"
#include "sg_internal.h"

namespace sg {

namespace {

constexpr int kQThreads = 256;
constexpr int kQMaxVecs = 16;  // vectors per thread: C <= 16 * 256 * 8 = 32768
constexpr int kQGroup = 4;     // blockscale: consecutive vectors a thread takes in one block

// Least integer e with amax <= 448 * 2^e, for finite amax > 0, by exact integer
// comparison: amax = M * 2^q, 448 = 7 * 2^6, so e = t - 6 + q with t the least
// integer such that 7 * 2^t >= M.
__device__ __forceinline__ int mx_exponent(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const uint32_t ef = (u >> 23) & 0xFFu;
  const uint64_t M = ef ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
  const int q = ef ? static_cast<int>(ef) - 150 : -149;
  int t = 0;
  if (M > 7) {
    // M has b bits, so 7 * 2^(b-3) < 2^b and 7 * 2^(b-2) >= 2^b > M: t is b-3 or b-2
    const int b = 32 - __clz(static_cast<uint32_t>(M));
    t = (7ull << (b - 3)) >= M ? b - 3 : b - 2;
  } else {
    while ((M << (1 - t)) <= 7) --t;
  }
  return t - 6 + q;
}

__device__ __forceinline__ float exp2_code(int code) {  // 2^(code - 127), code in [0, 254]
  return code > 0 ? __uint_as_float(static_cast<uint32_t>(code) << 23) : __uint_as_float(0x00400000u);
}

// The raw 16 (bf16) or 32 (fp32) bytes of one 8-element vector.
template <bool BF16>
struct Raw8 {
  uint4 w[BF16 ? 1 : 2];
};

template <bool BF16>
__device__ __forceinline__ void load_raw8(const void* X, int64_t elem, Raw8<BF16>& raw) {
  if constexpr (BF16) {
    raw.w[0] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(X) + elem));
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(X) + elem);
    raw.w[0] = __ldg(p);
    raw.w[1] = __ldg(p + 1);
  }
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const Raw8<BF16>& raw, float (&f)[8]) {
  if constexpr (BF16) {
    const uint32_t w[4] = {raw.w[0].x, raw.w[0].y, raw.w[0].z, raw.w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      f[4 * h + 0] = __uint_as_float(raw.w[h].x);
      f[4 * h + 1] = __uint_as_float(raw.w[h].y);
      f[4 * h + 2] = __uint_as_float(raw.w[h].z);
      f[4 * h + 3] = __uint_as_float(raw.w[h].w);
    }
  }
}

__device__ __forceinline__ uint2 cvt8(const float (&y)[8]) {
  uint32_t w[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t pair = __nv_cvt_float2_to_fp8x2(make_float2(y[2 * i], y[2 * i + 1]), __NV_SATFINITE, __NV_E4M3);
    w[i >> 1] |= (pair & 0xFFFFu) << (16 * (i & 1));
  }
  return make_uint2(w[0], w[1]);
}

// Eight codes of x / s (round to nearest even, saturated), s a power of two
// whose reciprocal inv_s is representable: x * inv_s is then the same correctly
// rounded value as x / s.
__device__ __forceinline__ uint2 quant8_pow2(const float (&f)[8], float inv_s) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = f[i] * inv_s;
  return cvt8(y);
}

// The correctly rounded quotient x / s without a division, by Markstein's method
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s), q = RN(x r), and
// twice q <- RN(q + (x - q s) r), each remainder x - q s exact in one fma, the
// second correction is RN(x / s) once r is correctly rounded and q within an ulp,
// barring underflow.  Here it is taken only for 2^-60 <= s <= 2^60: every quotient
// that can round to a nonzero e4m3 code (|x / s| >= 2^-11) then keeps its
// remainders normal, and smaller quotients round to +-0 either way.  A zero x
// would come out +0 from the corrections, so the sign of x is copied back (the
// quotient's sign is x's: s > 0).  Two lanes per packed fp32x2 instruction.
struct Recip {
  uint64_t r2;    // (r, r)
  uint64_t ns2;   // (-s, -s)
  bool fast;      // s in [2^-60, 2^60]
};

__device__ __forceinline__ Recip make_recip(float s) {
  const float r = __frcp_rn(s);
  Recip q;
  q.r2 = pack_f32x2(__float_as_uint(r), __float_as_uint(r));
  q.ns2 = pack_f32x2(__float_as_uint(-s), __float_as_uint(-s));
  q.fast = s >= 0x1p-60f && s <= 0x1p+60f;
  return q;
}

// Eight codes of x / s: the quotient correctly rounded in fp32 (the IEEE division
// where the scale is outside Markstein's range), then e4m3.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s, const Recip& rc) {
  float y[8];
  if (rc.fast) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = __float_as_uint(f[2 * i]), b = __float_as_uint(f[2 * i + 1]);
      const uint64_t x = pack_f32x2(a, b);
      uint64_t q = mul_f32x2(x, rc.r2);
      uint64_t e = fma_f32x2(q, rc.ns2, x);
      q = fma_f32x2(e, rc.r2, q);
      e = fma_f32x2(q, rc.ns2, x);
      q = fma_f32x2(e, rc.r2, q);
      float lo, hi;
      unpack_f32x2(q, lo, hi);
      y[2 * i] = __uint_as_float((__float_as_uint(lo) & 0x7FFFFFFFu) | (a & 0x80000000u));
      y[2 * i + 1] = __uint_as_float((__float_as_uint(hi) & 0x7FFFFFFFu) | (b & 0x80000000u));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(f[i], s);
  }
  return cvt8(y);
}

// Resident CTAs a launch sizes its registers for (0: the compiler's choice).
// mxfp8 on bf16 rows of 4 vectors a thread (4097 to 8192 elements) fits four
// CTAs an SM (64 registers, no spills) where the compiler alone takes three;
// an explicit bound elsewhere either spills or, at one CTA, lets ptpc and
// blockscale grow past three CTAs' registers.
template <int MODE, bool BF16, int VPT>
constexpr int q_min_ctas() {
  return (MODE == kModeMxfp8 && BF16 && VPT == 4) ? 4 : 0;
}

template <int MODE, bool BF16, int VPT>
__global__ void __launch_bounds__(kQThreads, (q_min_ctas<MODE, BF16, VPT>()))
    quantize_kernel(const void* __restrict__ X, uint8_t* __restrict__ Q, void* __restrict__ scale,
                    int R, int C) {
  __shared__ float red[kQThreads / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nvec = C / 8;
  // Vector i of this thread in the row.  ptpc and mxfp8: vectors tid, tid + 256,
  // ... (every load instruction of a warp reads 512 contiguous bytes).
  // blockscale: groups of kVB consecutive vectors, so a thread's group lies in
  // one 1x128 block (16 vectors), whose amax then needs 16 / kVB lanes, and the
  // scale's division and reciprocal are taken once per group instead of once per
  // vector.  Those two dominate the blockscale arithmetic; mxfp8's power-of-two
  // scale is cheap, and there the strided loads of groups cost more than they save.
  constexpr int kVB = (MODE == kModeBlockscale) ? (VPT < kQGroup ? VPT : kQGroup) : 1;
  static_assert(VPT % kVB == 0, "whole groups per thread");
  auto vidx = [&](int i) { return (i / kVB) * (kQThreads * kVB) + tid * kVB + (i % kVB); };
  // The next row's raw vectors are loaded while the current row is processed,
  // where they fit in 32 registers; otherwise each row is loaded when it starts.
  constexpr bool kPrefetch = VPT * (BF16 ? 4 : 8) <= 32;
  auto fetch = [&](Raw8<BF16> (&dst)[VPT], int rr) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = vidx(i);
      if (v < nvec && rr < R) load_raw8<BF16>(X, static_cast<int64_t>(rr) * C + 8 * static_cast<int64_t>(v), dst[i]);
    }
  };
  Raw8<BF16> next[kPrefetch ? VPT : 1];
  if constexpr (kPrefetch) fetch(next, blockIdx.x);
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int64_t row = static_cast<int64_t>(r) * C;
    float f[VPT][8];
    float local = 0.f;
    if constexpr (kPrefetch) {
      Raw8<BF16> raw[VPT];
#pragma unroll
      for (int i = 0; i < VPT; ++i) raw[i] = next[i];
      fetch(next, r + gridDim.x);
#pragma unroll
      for (int i = 0; i < VPT; ++i) unpack8<BF16>(raw[i], f[i]);
    } else {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = vidx(i);
        Raw8<BF16> raw;
        if (v < nvec) load_raw8<BF16>(X, row + 8 * static_cast<int64_t>(v), raw);
        unpack8<BF16>(raw, f[i]);
      }
    }
    // vectors past the row end (the last pass when C / 8 is not a multiple of
    // the block size) hold zeros
#pragma unroll
    for (int i = 0; i < VPT; ++i)
      if (vidx(i) >= nvec)
#pragma unroll
        for (int j = 0; j < 8; ++j) f[i][j] = 0.f;
    if constexpr (MODE == kModePtpc) {
#pragma unroll
      for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) local = fmaxf(local, fabsf(f[i][j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) local = fmaxf(local, __shfl_xor_sync(0xffffffffu, local, o));
      if (lane == 0) red[tid >> 5] = local;
      __syncthreads();
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
      const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      if (tid == 0) static_cast<float*>(scale)[r] = s;
      const Recip rc = make_recip(s);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = vidx(i);
        if (v < nvec) *reinterpret_cast<uint2*>(Q + row + 8 * static_cast<int64_t>(v)) = quant8(f[i], s, rc);
      }
      __syncthreads();  // red[] is reused by the next row
    } else {
      // a block is kBV consecutive vectors: the groups of kLanes consecutive lanes
      // of one warp (C is a multiple of the block, so a group is wholly inside
      // or wholly past the row)
      constexpr int kBV = MODE == kModeBlockscale ? 16 : 4;
      constexpr int kLanes = kBV / kVB;
      static_assert(kBV % kVB == 0, "a group inside one block");
#pragma unroll
      for (int g = 0; g < VPT / kVB; ++g) {
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < kVB; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[g * kVB + j][e]));
#pragma unroll
        for (int o = kLanes / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const int v0 = vidx(g * kVB);
        const bool live = v0 < nvec;
        const int blk = v0 / kBV;
        uint2 codes[kVB];
        if constexpr (MODE == kModeBlockscale) {
          const float s = a > 0.f ? __fdiv_rn(a, 448.0f) : 1.0f;
          if (live && (v0 % kBV) == 0) static_cast<float*>(scale)[static_cast<int64_t>(blk) * R + r] = s;
          const Recip rc = make_recip(s);
#pragma unroll
          for (int j = 0; j < kVB; ++j) codes[j] = quant8(f[g * kVB + j], s, rc);
        } else {
          int code = a > 0.f ? mx_exponent(a) + 127 : 127;
          code = code < 0 ? 0 : (code > 254 ? 254 : code);
          if (live && (v0 % kBV) == 0)
            static_cast<uint8_t*>(scale)[static_cast<int64_t>(blk) * R + r] = static_cast<uint8_t>(code);
          // 1/s = 2^(127 - code), code in [0, 254]: representable (normal or 2^-127)
          const float inv_s = exp2_code(254 - code);
#pragma unroll
          for (int j = 0; j < kVB; ++j) codes[j] = quant8_pow2(f[g * kVB + j], inv_s);
        }
        if (live) {
          uint8_t* dst = Q + row + 8 * static_cast<int64_t>(v0);  // 8 kVB-byte aligned
          if constexpr (kVB == 1) {
            *reinterpret_cast<uint2*>(dst) = codes[0];
          } else {
#pragma unroll
            for (int j = 0; j < kVB; j += 2)
              *reinterpret_cast<uint4*>(dst + 8 * j) =
                  make_uint4(codes[j].x, codes[j].y, codes[j + 1].x, codes[j + 1].y);
          }
        }
      }
    }
  }
}

template <int MODE, bool BF16, int VPT>
sg_status_t launch_q(const void* X, uint8_t* Q, void* S, int R, int C, int grid, cudaStream_t st) {
  quantize_kernel<MODE, BF16, VPT><<<grid, kQThreads, 0, st>>>(X, Q, S, R, C);
  return launch_status();
}

template <int MODE, bool BF16>
sg_status_t launch_q_vpt(const void* X, uint8_t* Q, void* S, int R, int C, int grid, cudaStream_t st) {
  const int vecs = (C / 8 + kQThreads - 1) / kQThreads;
  if (vecs <= 1) return launch_q<MODE, BF16, 1>(X, Q, S, R, C, grid, st);
  if (vecs <= 2) return launch_q<MODE, BF16, 2>(X, Q, S, R, C, grid, st);
  if (vecs <= 4) return launch_q<MODE, BF16, 4>(X, Q, S, R, C, grid, st);
  if (vecs <= 8) return launch_q<MODE, BF16, 8>(X, Q, S, R, C, grid, st);
  return launch_q<MODE, BF16, 16>(X, Q, S, R, C, grid, st);
}

template <int MODE>
sg_status_t launch_q_mode(bool bf16, const void* X, uint8_t* Q, void* S, int R, int C, int grid,
                          cudaStream_t st) {
  return bf16 ? launch_q_vpt<MODE, true>(X, Q, S, R, C, grid, st)
              : launch_q_vpt<MODE, false>(X, Q, S, R, C, grid, st);
}

}  // namespace

int64_t quantize_max_cols() { return static_cast<int64_t>(kQMaxVecs) * kQThreads * 8; }

sg_status_t quantize_launch(int mode, bool bf16, const void* X, int64_t R, int64_t C, void* Q,
                            void* scale, int num_sms, cudaStream_t st) {
  const int r = static_cast<int>(R), c = static_cast<int>(C);
  const int64_t g = R < static_cast<int64_t>(num_sms) * 8 ? R : static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(g);
  uint8_t* q = static_cast<uint8_t*>(Q);
  switch (mode) {
    case kModePtpc: return launch_q_mode<kModePtpc>(bf16, X, q, scale, r, c, grid, st);
    case kModeBlockscale: return launch_q_mode<kModeBlockscale>(bf16, X, q, scale, r, c, grid, st);
    case kModeMxfp8: return launch_q_mode<kModeMxfp8>(bf16, X, q, scale, r, c, grid, st);
  }
  return SG_ERR_INVALID_ARG;
}

}  // namespace sg
