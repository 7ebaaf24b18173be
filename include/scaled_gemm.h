/*
 * scaled_gemm.h -- C ABI of the GB300 (sm_103a) scaled FP8 / BF16 GEMM library
 * (libscaledgemm.so).
 *
 * The operation (one launch):
 *
 *     C[M,N] = bf16( (A[M,K] . B[N,K]^T) (.) scales ),   fp32 accumulation,
 *
 * in one of four modes:
 *
 *   SG_MODE_PTPC        per-token x per-channel:  C = bf16(acc[m,n] * a_scale[m] * b_scale[n]).
 *                       ROCm/mori PR 809, "Using it" (A [M,K] fp8 with a per-row scale from
 *                       quantize_per_token, the weight shard B [N,K] with its scale,
 *                       bf16 [M,N] out); ROCm/mori PR 785 cost table ("ptpc").
 *   SG_MODE_BLOCKSCALE  fp32 scales per 1x128 block of A and per 128x128 block of B:
 *                       C = bf16( sum_j acc_j[m,n] * a_scale[j][m] * b_scale[n/128][j] ),
 *                       acc_j the fp32 partial over K block j.  ROCm/mori PR 785 cost table
 *                       ("blockscale"); PR 809 "Not done yet" (the A scale is K-block major).
 *   SG_MODE_MXFP8       e8m0 scales per 32 consecutive K elements of each row of A and B:
 *                       C = bf16( sum_j acc_j * 2^(a_scale[j][m]-127) * 2^(b_scale[j][n]-127) ).
 *                       ROCm/mori PR 785 cost table ("mxfp8") and Scope.
 *   SG_MODE_BF16        plain GEMM: C = bf16(acc).  deepseek-ai/DeepGEMM PR 453, Summary and
 *                       Reproduction (BF16 GEMM, fp32 accumulation).
 *
 * Element types: fp8 is e4m3fn (OCP OFP8: bias 7, no infinities, max 448), bf16 is
 * the upper half of an IEEE binary32, e8m0 is an unsigned biased exponent (bias 127,
 * 255 = NaN).  Rounding to bf16 is round-to-nearest-even.
 *
 * Memory layout (every pointer is a DEVICE pointer, owned by the caller, never
 * retained by the library after the launch returns, 16-byte aligned):
 *   A        [M][K] row-major (K contiguous): e4m3 bytes, or bf16 in SG_MODE_BF16
 *   B        [N][K] row-major (K contiguous): same element type as A
 *   C        [M][N] row-major bf16 (N contiguous); must not overlap A, B or the scales
 *            (checked on the host: an overlap returns SG_ERR_INVALID_ARG)
 *   ptpc        a_scale float[M],            b_scale float[N]
 *   blockscale  a_scale float[K/128][M],     b_scale float[ceil(N/128)][K/128]
 *   mxfp8       a_scale uint8[K/32][M],      b_scale uint8[K/32][N]     (e8m0 codes)
 *   bf16        a_scale = b_scale = NULL
 *
 * Shape rules (checked on the host before anything is launched):
 *   0 <= M <= M_max (M == 0 or N == 0 launches nothing), N % 16 == 0,
 *   K % 16 == 0 (ptpc), K % 8 == 0 (bf16), K % 128 == 0 (blockscale),
 *   K % 32 == 0 (mxfp8), M, N, K < 2^31.  K == 0 writes C = 0.
 *
 * Errors: every call returns an sg_status_t and never aborts or prints (set the
 * environment variable SG_DEBUG=1 to log rejected calls to stderr).  Kernel faults,
 * like any CUDA asynchronous error, surface at the caller's next synchronisation.
 *
 * Streams: scaled_gemm_launch is asynchronous on `stream` and never synchronises.
 * A ptpc, blockscale or bf16 handle is immutable after creation, so launches on one
 * such handle from several host threads or streams are safe.  An mxfp8 handle owns
 * a device workspace (its launch first rearranges the scales there for the tensor
 * core), so launches on one mxfp8 handle must be ordered: issue them on one stream,
 * or order their streams, or use one handle per stream.  (The one departure from a
 * workspace-free plan: the block-scaled MMA reads its scales from tensor memory in
 * a layout the K-block-major scale arrays do not have.)  Destroying a handle must
 * not race a launch on it.
 *
 * Every kernel is launched with programmatic stream serialization: it may be
 * scheduled while the kernel before it on `stream` is still running, sets up its
 * barriers and tensor memory, and then waits (griddepcontrol.wait) until that kernel
 * has completed and its memory writes are visible before it reads or writes any
 * global memory.  Launches on one stream therefore see each other's results exactly
 * as plain stream-ordered launches do; only the set-up overlaps.
 */
#ifndef SCALED_GEMM_H
#define SCALED_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; the same type as cudaStream_t.  NULL = the legacy default stream. */
typedef struct CUstream_st* sg_stream_t;

/* Opaque GEMM plan, owned by the library. */
typedef struct sg_gemm* sg_handle_t;

typedef enum {
    SG_MODE_BF16 = 0,
    SG_MODE_PTPC = 1,
    SG_MODE_BLOCKSCALE = 2,
    SG_MODE_MXFP8 = 3
} sg_mode_t;

typedef enum {
    SG_OK = 0,
    SG_ERR_INVALID_ARG = 1,        /* NULL handle/pointer, bad mode, M > M_max, negative size */
    SG_ERR_UNSUPPORTED_SHAPE = 2,  /* N, K or M break the shape rules above */
    SG_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
    SG_ERR_UNSUPPORTED_DEVICE = 4, /* the device is not compute capability 10.3 (sm_103a) */
    SG_ERR_CUDA = 5,               /* a CUDA runtime / driver call failed */
    SG_ERR_TIMEOUT = 6             /* a kernel wait ran past its time limit (see debug_status) */
} sg_status_t;

/* Create a plan for one (mode, N, K) that serves any M <= M_max on `device`
 * (-1 = the current device).  The plan holds a 16-byte device status word, set
 * up here, that kernels write only when a wait times out; an mxfp8 plan also
 * allocates here its scale workspace, (ceil(M_max/128) + 8 ceil(N/224)) *
 * ceil(K/128) * 512 bytes of device memory.
 * On success *out receives the handle; on failure *out is set to NULL.
 * Cited: ROCm/mori PR 809, "Using it" (one instance serves one (n, k) and any M
 * up to m_max; bad configuration is refused at construction).                   */
sg_status_t scaled_gemm_create(sg_handle_t* out, int mode, int64_t N, int64_t K, int64_t M_max,
                               int device);

/* Launch C = op(A, B, a_scale, b_scale) for M rows on `stream` (see the layout and
 * shape rules above).  The call validates its arguments, builds the TMA
 * descriptors on the host and enqueues one persistent kernel; it never blocks.
 * Cited: ROCm/mori PR 809, "Using it" (op(a_fp8, b, a_scale, b_scale, out=));
 * ROCm/aiter PR 6539, Test Plan (run_torch(xq, wq, x_scale, w_scale)).          */
sg_status_t scaled_gemm_launch(sg_handle_t h, const void* A, const void* B, const void* a_scale,
                               const void* b_scale, void* C, int64_t M, sg_stream_t stream);

/* Gather-GEMM on a ptpc plan: output row i (0 <= i < M) is the ptpc GEMM row of
 * source row idx[i] of A_src, scaled by a_scale_src[idx[i]] and b_scale[n]:
 *   C[i][n] = bf16( (sum_k A_src[idx[i]][k] * B[n][k]) * a_scale_src[idx[i]] * b_scale[n] )
 * A_src e4m3 [R][K] row-major, a_scale_src float[R], idx int32[M] (device
 * pointers, 16-byte aligned, caller-owned); B, b_scale and C as for ptpc.  An index
 * outside [0, R) names no row: that output row is zero (never read out of
 * bounds).  The rows are gathered inside the GEMM's pipeline: two warps of each
 * CTA copy every stage's rows with cp.async into the swizzled shared-memory tile
 * the MMA reads; they are never copied out first.  Shape rules as for ptpc, with
 * 0 <= R < 2^31; R == 0 or K == 0 writes C = 0.  Returns SG_ERR_INVALID_ARG on a plan of another mode.
 * Cited: ROCm/aiter PR 6539, Motivation and Technical Details (gather_kv_b_proj:
 * the KV projection GEMM over rows gathered by index).                            */
sg_status_t scaled_gemm_launch_gather(sg_handle_t h, const void* A_src, int64_t R, const int32_t* idx,
                                      const void* B, const void* a_scale_src, const void* b_scale,
                                      void* C, int64_t M, sg_stream_t stream);

/* Release the plan (its status word and, for mxfp8, its workspace).  NULL is
 * accepted.  Must not race a launch being enqueued on the same handle from another
 * thread; launches already enqueued may still run (freeing device memory waits for
 * the device first).  Returns SG_OK,
 * or SG_ERR_CUDA if freeing device memory failed (the handle is released anyway).
 * Cited: ROCm/mori PR 809, "Using it" (the op is an instance used inside a
 * `with` block that releases it at the end) and "Test plan" (close).            */
sg_status_t scaled_gemm_destroy(sg_handle_t h);

/* A static English description of a status code (never NULL; an unknown code
 * gives "unknown status").  Refusals are returned, not raised, so that a C caller
 * sees them: ROCm/mori PR 809, "Using it" (operands the launch would misread are
 * refused with an error; the constructor refuses bad configuration).           */
const char* scaled_gemm_status_string(sg_status_t s);

/* Tile geometry of a launch at M = M_max: BM x BN output tiles per CTA (BN: the
 * tile's columns; CTA pairs share a BN-wide tile), BK elements of K per pipeline
 * stage, `stages` shared-memory stages, `grid` persistent CTAs (whole clusters,
 * where the kernel runs CTAs in pairs).  mxfp8, ptpc and bf16 choose BN per launch
 * from M and N (see scaled_gemm_set_tile), so a smaller M may use the other width.  Any output
 * pointer may be NULL.  Returns SG_ERR_INVALID_ARG for a NULL handle.
 * Cited: a review of ROCm/mori PR 809, Smaller points (the tile configuration a
 * kernel serves is validated and reported, and the default should follow the
 * shape).                                                                        */
sg_status_t scaled_gemm_get_config(sg_handle_t h, int* bm, int* bn, int* bk, int* stages, int* grid);

/* Pin the output-tile width every later launch of the plan uses, or pass 0 to let
 * each launch choose (the default).  mxfp8 has two widths: 224 (256 x 224 tiles per
 * CTA pair) and 128 (256 x 128, the narrow mxfp8 tile ROCm/mori PR 785 names in its
 * Test section); a launch chooses 128 where 224-wide tiles would leave pairs of SMs
 * idle (small M), by an estimate of waves of tiles x width (the shape-aware default
 * a review of ROCm/mori PR 809, Smaller points, asks for).
 * ptpc and bf16 have two widths: 256 (256 x 256 tiles per CTA pair) and 128,
 * chosen the same way (128 only where fewer 256-wide tiles than pairs of SMs
 * exist, e.g. one row panel at M <= 256); the gather launch always uses its one
 * 256-wide tile.  blockscale has one width (256) and accepts only 0 or 256.  The
 * two widths of a mode sum every output element over K in the same order of MMA
 * instructions, so they give the same bits.
 * Not to be called while a launch of the plan is being enqueued from another
 * thread.
 * Returns SG_ERR_INVALID_ARG for a NULL handle or a width the mode does not have. */
sg_status_t scaled_gemm_set_tile(sg_handle_t h, int bn);

/* Read and clear the plan's device status word: synchronises `stream`, then stores
 * SG_OK or SG_ERR_TIMEOUT in *code and, for a timeout, the role / wait site that gave
 * up in *where (0 otherwise).  Every mbarrier wait in the kernels is bounded; on
 * expiry the kernel records the site here, drains its own copies in flight, frees
 * its tensor memory and returns, so the context stays usable.  Returns
 * SG_ERR_INVALID_ARG for a NULL handle or code, SG_ERR_CUDA if the copy fails.
 * Cited: ROCm/mori PR 809, Worth a reviewer's attention (a grid whose blocks all
 * spin on data that never arrives never finishes): here no wait is unbounded, and
 * a wait that gives up is reported instead of hanging the stream.               */
sg_status_t scaled_gemm_debug_status(sg_handle_t h, sg_stream_t stream, int32_t* code,
                                     int32_t* where);

/* Set the time limit of every kernel-side wait for this plan (nanoseconds; 0 = the
 * default, 4 s) and, for tests of the watchdog only, make the producer of every CTA
 * skip its `skip_kstep`-th pipeline stage (-1 = never) so that the consumer's wait
 * expires.  Not for production use.  Returns SG_ERR_INVALID_ARG for a NULL handle,
 * a negative limit or skip_kstep < -1.  Cited: ROCm/aiter PR 6539, Technical
 * Details (the races were hunted with fault injection); the fault here is made on
 * the host's side of the launch, never by corrupting device memory.             */
sg_status_t scaled_gemm_set_debug(sg_handle_t h, int64_t timeout_ns, int64_t skip_kstep);

/* Element types of the activations given to scaled_gemm_quantize. */
typedef enum { SG_DTYPE_BF16 = 0, SG_DTYPE_F32 = 1 } sg_dtype_t;

/* The step before the GEMM: quantise X [R][C] (row-major; bf16 or fp32 per
 * x_dtype; finite values) to e4m3 codes Q [R][C] and scales in the A-side layout
 * of `mode`:
 *   SG_MODE_PTPC        scale float[R]         one per row (per token)
 *   SG_MODE_BLOCKSCALE  scale float[C/128][R]  one per 1 x 128 block, K-block major
 *   SG_MODE_MXFP8       scale uint8[C/32][R]   e8m0, one per 32 elements, K-block major
 * For a row segment with amax = max |x|: ptpc / blockscale s = amax / 448 (one fp32
 * IEEE division; 1 if amax == 0); mxfp8 e = the least integer with amax <= 448 * 2^e
 * (0 if amax == 0), code = clamp(e + 127, 0, 254), s = 2^(code - 127).  Every code is
 * q = e4m3(x / s): one fp32 IEEE division, then round to nearest even, saturated to
 * +-448.  Shape rules: C % 16 == 0 (ptpc), C % 128 (blockscale), C % 32 (mxfp8),
 * C <= 32768; pointers 16-byte aligned, device memory, caller-owned.  Asynchronous
 * on `stream`.  Cited: ROCm/mori PR 809, "Using it" (a_fp8, a_scale =
 * quantize_per_token(x) before the GEMM) and "Not done yet" (blockscale / mxfp8 A
 * scales are K-block major).                                                    */
sg_status_t scaled_gemm_quantize(int mode, int x_dtype, const void* X, int64_t R, int64_t C, void* Q,
                                 void* scale, sg_stream_t stream);

/* ptpc GEMM for callers that cannot allocate device memory.  (The paper has no
 * counterpart: this entry point belongs to this library's interface only.)
 *
 * scaled_gemm_create allocates the kernel's 16-byte watchdog status record with
 * cudaMalloc, which some callers cannot do: code running inside a custom
 * allocator or a memory-pool callback (where a nested cudaMalloc would re-enter
 * the allocator), or processes whose device memory is all reserved up front by a
 * pool that owns every allocation.  This call needs no handle and allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine): the status record lives in a
 * 64-byte static device array inside the library, which every GPU that loads
 * the library holds until the process exits.  A launch that would need more
 * scratch than that array holds is rejected with SG_ERR_UNSUPPORTED_SHAPE.
 *
 * Operands, layouts and shape rules are those of SG_MODE_PTPC above, with M, N, K
 * given directly (K == 0 is rejected; use scaled_gemm_launch).  The current
 * device is used.  The first call on a device sets it up (checks compute
 * capability 10.3, looks up the array's device address, sets the kernel's
 * shared-memory limit); make that first call before any stream capture.  Every
 * call clears the shared status record on `stream` before its kernel and the
 * record keeps the last call's contents; calls whose kernels overlap on the GPU
 * race on it, so serialise them (one stream) if the record matters.  The record
 * cannot be read through this entry point; use the handle API to diagnose a
 * watchdog timeout.                                                              */
sg_status_t scaled_gemm_launch_noalloc(const void* A, const void* B, const void* a_scale,
                                       const void* b_scale, void* C, int64_t M, int64_t N,
                                       int64_t K, sg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SCALED_GEMM_H */
