/*
 * sk.h -- C ABI of libsk.so: the small-M skinny GEMM with a deterministic
 * split-K reduction and its two fused epilogues, for NVIDIA GB300 (sm_103a).
 *
 * Source of the operations (vLLM API pages of the Muse Spark specialized
 * decode package; each entry point below cites its passage by page title and
 * section):
 *   cutedsl/gemm/unpooler      -- module docstring, Unpooler, launch_unsupported
 *   cutedsl/moe/pooler_gather  -- module docstring, Pooler, PoolerLayer,
 *                                 nvfp4_compute_output_scale, cvt_* helpers
 *   cutedsl/oproj/batt         -- AttentionBoundary, OProjection
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers unless a comment says otherwise. Tensors are
 *     contiguous and row-major; BF16 tensors are passed as raw 16-bit words.
 *     Every tensor pointer must be 16-byte aligned.
 *   - The caller owns every buffer. No call allocates device or host memory,
 *     no call synchronizes, and no call compiles anything: each one only
 *     validates its arguments on the host and enqueues kernels on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream). The calls other
 *     than sk_gemm_rmsnorm_nvfp4_static can be captured into a CUDA graph once
 *     the device has been used by the library (first call does one-time
 *     per-device set-up of kernel attributes).
 *   - Kernels are chained with programmatic dependent launch: weights (which
 *     no kernel writes) are read before a kernel waits for its predecessor in
 *     the stream; activations are read, and outputs written, only after it.
 *   - BF16 outputs never hold -0.0: a negative zero is stored as +0.0.
 *   - Results depend only on the inputs and the launch shape (m, n, k and the
 *     split count): repeated calls give bitwise-identical outputs.
 *   - Errors: invalid arguments are rejected on the host before any launch,
 *     with a status code and a message from sk_last_error(). A device that is
 *     not compute capability 10.3 returns SK_ERR_ARCH. Launch failures return
 *     SK_ERR_CUDA. A kernel never traps: every wait inside a kernel is
 *     bounded, and a wait that runs out sets a bit in the library's device
 *     status word (read it with sk_device_status) and the kernel returns.
 */
#ifndef SK_H_
#define SK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SK_VERSION 1
#define SK_MAX_M 16 /* token rows per call */

typedef enum sk_status {
    SK_OK = 0,
    SK_ERR_INVALID_ARG = 1,    /* null pointer, bad shape, misalignment     */
    SK_ERR_UNSUPPORTED = 2,    /* shape valid but no launch (split count)   */
    SK_ERR_ARCH = 3,           /* current device is not compute capability 10.3 */
    SK_ERR_WORKSPACE = 4,      /* workspace too small                        */
    SK_ERR_CUDA = 5,           /* CUDA runtime error (message has details)   */
    SK_ERR_DEVICE_TIMEOUT = 6  /* a bounded device-side wait ran out         */
} sk_status;

/* Device status bits (sk_device_status). */
#define SK_DEVICE_WAIT_PRODUCER 0x1u /* weight/activation copy never landed */
#define SK_DEVICE_WAIT_MMA 0x2u      /* tensor-core stage never filled      */
#define SK_DEVICE_WAIT_EPILOGUE 0x4u /* accumulator never completed         */
#define SK_DEVICE_WAIT_PROBE 0x10u   /* sk_wait_probe's wait ran out (expected) */
#define SK_DEVICE_WAIT_TEARDOWN 0x20u /* after an abort, the MMAs never quiesced before TMEM release */

/* Message of the last failed call on this host thread ("" if none). The
   string lives in thread-local storage owned by the library. */
const char *sk_last_error(void);

/* SK_VERSION of the built library. */
int sk_version(void);

/* Number of splits of K the GEMM uses for (m, n, k, splits): `splits` itself
   when it is 1, 2, 4, 8 or 16, else (splits == 0) the automatic choice for the
   current device. Returns 0 and sets sk_last_error() when the shape has no
   launch. Host-only; the automatic choice queries the current device. */
int sk_gemm_splits(int m, int n, int k, int splits);

/* Why (m, n, k, splits) has no launch, or SK_OK. Mirrors the unpooler page's
   launch_unsupported and Unpooler.unsupported: 1 <= m <= 16, n > 0 with
   n % 16 == 0, k > 0 with k % (64 * S) == 0 for the split count S, and
   S in {0 (auto), 1, 2, 4, 8, 16}. Host-only, launches nothing. */
sk_status sk_gemm_supported(int m, int n, int k, int splits);

/*
 * sk_gemm_bf16 -- y[m, n] = bf16_rn( sum_k x[m, k] * w[n, k] )
 * (cutedsl/gemm/unpooler, module docstring and Unpooler.run; the same product
 * serves the pooler GEMM of cutedsl/moe/pooler_gather and the o_proj of
 * cutedsl/oproj/batt, OProjection).
 *   x  BF16 [m, k] activations, 1 <= m <= 16
 *   w  BF16 [n, k] weight, row-major (each output feature's K values contiguous)
 *   y  BF16 [m, n] output (written, never read)
 *   splits  0 for the automatic choice, or 1, 2, 4, 8, 16: the K range is cut
 *           into `splits` equal slices reduced in a fixed order on chip.
 * Products are exact, accumulation is FP32 on the tensor cores, the split
 * partials are summed in FP32 in split order, and the sum is rounded once to
 * BF16 (nearest, ties to even).
 */
sk_status sk_gemm_bf16(const void *x, const void *w, void *y, int m, int n, int k,
                       int splits, void *stream);

/* Flags of sk_gemm_bf16_ex. */
#define SK_GEMM_X_READY 0x1u /* no kernel still running may write x */

/*
 * sk_gemm_bf16_ex -- sk_gemm_bf16 with flags. This library's kernels start
 * before the kernel ahead of them on the stream has finished (programmatic
 * dependent launch): they stream their weights at once, read their
 * activations only after that kernel completes, and complete only after it.
 * With SK_GEMM_X_READY the GEMM reads x at once as well; only its stores of y
 * wait, so y is still written in stream order. The caller promises that no
 * kernel that writes x can still be running when the GEMM starts. That holds
 * when x was written by host copies only, or by kernels that precede a copy,
 * an event wait, a launch without programmatic dependent launch, or a host
 * synchronisation on this stream. It does not hold for a kernel just ahead in
 * a chain of this library's calls, nor for any call that chain reaches back
 * to. A run of GEMMs on one such input (rotated weights, several projections
 * of the same activations) then overlaps call with call. No counterpart on the
 * pages: there, activations are always read after the wait (unpooler page,
 * module docstring). Results are those of sk_gemm_bf16, bit for bit.
 *   flags: 0 or SK_GEMM_X_READY; other bits are rejected (SK_ERR_INVALID_ARG).
 */
sk_status sk_gemm_bf16_ex(const void *x, const void *w, void *y, int m, int n, int k,
                          int splits, unsigned flags, void *stream);

/*
 * sk_gemm_prefetch_next -- a hint for the next GEMM that this host thread
 * enqueues (sk_gemm_bf16, sk_gemm_rmsnorm_nvfp4, sk_gemm_rmsnorm_bf16,
 * sk_gemm_dual_norm): once each of its CTAs has issued the copies of its own
 * weight slice, it starts towards L2 the first weight stages of the GEMM
 * y' = x' @ w_next^T (w_next BF16 [n_next, k_next], automatic splits) that
 * follows it in the stream, so that HBM keeps streaming through the first
 * GEMM's drain and epilogue, whatever runs between the two, and the second's
 * launch. No counterpart on the pages (there, each call streams only its own
 * weight). Results are unchanged; only timing depends on the hint.
 *   w_next 16-byte aligned, (n_next, k_next) a supported GEMM shape;
 *   w_next NULL clears a pending hint. The next GEMM enqueue on this thread
 *   consumes the hint (thread-local state); a call that fails before its GEMM
 *   is enqueued leaves it pending. A hint whose GEMM is later run with explicit
 *   splits other than the automatic ones warms the wrong tiles: still correct.
 */
sk_status sk_gemm_prefetch_next(const void *w_next, int n_next, int k_next);

/*
 * sk_rmsnorm_nvfp4 -- pre-expert RMSNorm of a BF16 [m, n] input, then NVFP4
 * (cutedsl/moe/pooler_gather: module docstring, PoolerLayer, pooler_layer,
 * nvfp4_compute_output_scale, cvt_e2m1x8_f32, cvt_f32_to_e4m3).
 *   r[i]    = 1 / sqrt( sum_j y[i,j]^2 / n + eps )                (FP32)
 *   z[i,j]  = bf16_rn( y[i,j] * r[i] * (norm_w[j] + gain_center) )
 *   per block of 16 columns b:
 *     amax  = max |z|,  sf = e4m3_rn_satfinite( (amax / 6) * gs )
 *     os    = sf == 0 ? 0 : 1 / (float(sf) * (1 / gs))           (IEEE FP32)
 *     code  = e2m1_rn_satfinite( z * os )
 *   a[i, j/2]   : code of column 2c in the low nibble, 2c + 1 in the high nibble
 *   a_sf[i, b]  : float8_e4m3fn bits, row-major, not swizzled
 *   y       BF16 [m, n], 1 <= m <= 16, n % 16 == 0, 16 <= n <= 16384
 *   norm_w  BF16 [n];  global_scale: device FP32 [1]
 *   a       u8 [m, n/2];  a_sf u8 [m, n/16];  z_out BF16 [m, n] or NULL
 */
sk_status sk_rmsnorm_nvfp4(const void *y, const void *norm_w, float eps, float gain_center,
                           const float *global_scale, uint8_t *a, uint8_t *a_sf, void *z_out,
                           int m, int n, void *stream);

/*
 * sk_rmsnorm_bf16 -- pre-expert RMSNorm of a BF16 edge layer: the rows the
 * experts take in BF16 instead of NVFP4 (cutedsl/moe/pooler_gather, module
 * docstring, "BF16 edge layers" / ExpertsInputBf16, and the ExpertNorm launch
 * in Pooler's edge-layer path). Same norm as sk_rmsnorm_nvfp4's z:
 *   z = bf16(y * rsqrt(mean(y^2) + eps) * (norm_w + gain_center)), -0 -> +0.
 *   y BF16 [m, n], norm_w BF16 [n], z BF16 [m, n]; 1 <= m <= 16, n a multiple
 *   of 16 in [16, 16384]; all pointers 16-byte aligned.
 */
sk_status sk_rmsnorm_bf16(const void *y, const void *norm_w, float eps, float gain_center, void *z,
                          int m, int n, void *stream);

/*
 * sk_gemm_rmsnorm_bf16 -- the pooler for a BF16 edge layer: y = x @ w^T (as
 * sk_gemm_bf16, into the workspace), then sk_rmsnorm_bf16 of y into z
 * (cutedsl/moe/pooler_gather, Pooler.run for a layer without a global scale:
 * it returns the normalised BF16 rows). Workspace: at least
 * sk_gemm_rmsnorm_nvfp4_workspace(m, n) bytes, 256-byte aligned; it holds y
 * on return. Constraints are those of sk_gemm_bf16 and sk_rmsnorm_bf16.
 */
sk_status sk_gemm_rmsnorm_bf16(const void *x, const void *w, const void *norm_w, float eps,
                               float gain_center, void *z, void *workspace,
                               size_t workspace_bytes, int m, int n, int k, int splits,
                               void *stream);

/* Size in bytes of the workspace sk_gemm_rmsnorm_nvfp4 needs for (m, n): the
   BF16 GEMM output that the norm reads back (m * n * 2, rounded up to 256). */
size_t sk_gemm_rmsnorm_nvfp4_workspace(int m, int n);

/*
 * sk_gemm_rmsnorm_nvfp4 -- the pooler: y = x @ w^T (as sk_gemm_bf16, into the
 * workspace), then sk_rmsnorm_nvfp4 of y (cutedsl/moe/pooler_gather, module
 * docstring and Pooler.run for an NVFP4 layer, on one GPU).
 *   x BF16 [m, k], w BF16 [n, k], norm_w BF16 [n], global_scale device FP32 [1]
 *   a u8 [m, n/2], a_sf u8 [m, n/16], z_out BF16 [m, n] or NULL
 *   workspace: device buffer of at least sk_gemm_rmsnorm_nvfp4_workspace(m, n)
 *   bytes, 256-byte aligned; its contents on return are the GEMM output y.
 * Constraints are those of sk_gemm_bf16 and sk_rmsnorm_nvfp4 together.
 */
sk_status sk_gemm_rmsnorm_nvfp4(const void *x, const void *w, const void *norm_w, float eps,
                                float gain_center, const float *global_scale, uint8_t *a,
                                uint8_t *a_sf, void *z_out, void *workspace,
                                size_t workspace_bytes, int m, int n, int k, int splits,
                                void *stream);

/*
 * sk_nvfp4_quantize -- the NVFP4 step alone: BF16 z [m, n] -> a, a_sf with the
 * same block arithmetic and byte layout as sk_rmsnorm_nvfp4 (same device code).
 * 1 <= m, n % 16 == 0.
 */
sk_status sk_nvfp4_quantize(const void *z, const float *global_scale, uint8_t *a,
                            uint8_t *a_sf, int m, int n, void *stream);

/*
 * sk_dual_norm_residual -- the attention boundary on one GPU
 * (cutedsl/oproj/batt, AttentionBoundary.run without the all-reduce):
 *   r1[i]   = 1 / sqrt( sum_j p[i,j]^2 / h + eps_post )
 *   q[i,j]  = p[i,j] * r1[i] * (post_w[j] + gc_post)    (q = p * r1 if post_w == NULL)
 *   s[i,j]  = alpha * s[i,j] + beta[j] * q[i,j]          (FP32, in place)
 *   r2[i]   = 1 / sqrt( sum_j s[i,j]^2 / h + eps_pre )    (over the updated s)
 *   out[i,j]= bf16_rn( s[i,j] * r2[i] * (pre_w[j] + gc_pre) )
 *   partial BF16 [m, h]; resid FP32 [m, h] (read and written); post_w BF16 [h]
 *   or NULL; beta, pre_w BF16 [h]; out BF16 [m, h].
 *   1 <= m <= 16, h % 8 == 0, 8 <= h <= 8192. All arithmetic is FP32.
 */
sk_status sk_dual_norm_residual(const void *partial, float *resid, const void *post_w,
                                float alpha, const void *beta, const void *pre_w, void *out,
                                float eps_post, float eps_pre, float gc_post, float gc_pre,
                                int m, int h, void *stream);

/* Size in bytes of the workspace sk_gemm_dual_norm needs: the BF16 partial
   [m, n] (m * n * 2, rounded up to 256). */
size_t sk_gemm_dual_norm_workspace(int m, int n);

/*
 * sk_gemm_dual_norm -- o_proj then the attention boundary: partial = x @ w^T
 * (as sk_gemm_bf16, into the workspace), then sk_dual_norm_residual of the
 * partial (cutedsl/oproj/batt, OProjection.run followed by
 * AttentionBoundary.run, on one GPU). Arguments as in the two calls it chains,
 * with h = n.
 */
sk_status sk_gemm_dual_norm(const void *x, const void *w, float *resid, const void *post_w,
                            float alpha, const void *beta, const void *pre_w, void *out,
                            float eps_post, float eps_pre, float gc_post, float gc_pre,
                            void *workspace, size_t workspace_bytes, int m, int n, int k,
                            int splits, void *stream);

/*
 * sk_gemm_nvfp4w_bf16 -- weight-only NVFP4 GEMM:
 *   y[m, n] = bf16_rn( w_scale * sum_k x[m, k] * W[n, k] ),
 *   W[n, k] = e2m1(code[n, k]) * e4m3(wsf[n, k / 16])
 * No counterpart on the pages: the weight is held in the NVFP4 byte layout that
 * cutedsl/moe/pooler_gather (module docstring) gives for the experts' input,
 * applied to the rows of W along K, so the GEMM streams 4.5 bits per weight
 * instead of 16. sk_nvfp4_quantize of a BF16 weight [n, k] with global scale
 * gs produces (wq, wsf), with w_scale = 1 / gs.
 *   x        BF16 [m, k] activations, 1 <= m <= 16
 *   wq       u8 [n, k/2]: e2m1 codes, column 2c in the low nibble, 2c+1 high
 *   wsf      u8 [n, k/16]: float8_e4m3fn scale of each 16 columns of a row,
 *            row-major, not swizzled (NaN encodings are out of contract)
 *   w_scale  device FP32 [1], multiplies the sum (read after the kernel ahead
 *            in the stream completes)
 *   y        BF16 [m, n] output; -0.0 is stored as +0.0
 *   n % 16 == 0, k % 256 == 0, splits 0 (automatic) or 1, 2, 4, 8, 16 with
 *   k % (256 * splits) == 0; x, wq, wsf, y 16-byte aligned.
 * Each weight is expanded exactly to BF16 on chip (code * scale has at most
 * six significant bits); the products are accumulated in FP32 on the tensor
 * cores, the split partials summed in split order, the sum multiplied by
 * w_scale in FP32 and rounded once to BF16. Bitwise reproducible for a given
 * (m, n, k, splits).
 */
sk_status sk_gemm_nvfp4w_bf16(const void *x, const uint8_t *wq, const uint8_t *wsf,
                              const float *w_scale, void *y, int m, int n, int k, int splits,
                              void *stream);

/* Why (m, n, k, splits) has no weight-only NVFP4 GEMM launch, or SK_OK
   (host-only). */
sk_status sk_gemm_nvfp4w_supported(int m, int n, int k, int splits);

/* Split count the weight-only NVFP4 GEMM uses for (m, n, k, splits) on the
   current device (splits itself when nonzero); 0 if the shape has no launch. */
int sk_gemm_nvfp4w_splits(int m, int n, int k, int splits);

/* Bytes of the static device scratch behind sk_gemm_rmsnorm_nvfp4_static:
   room for a BF16 [m, n] GEMM output with m * n <= 131072 (16 x 8192). */
#define SK_STATIC_SCRATCH_BYTES (16u * 8192u * 2u)

/*
 * sk_gemm_rmsnorm_nvfp4_static -- sk_gemm_rmsnorm_nvfp4 without a workspace
 * argument, for callers that cannot allocate device memory: an inference-
 * engine plugin whose enqueue function is handed no workspace, or a serving
 * loop whose memory is budgeted once at start-up. The pages have no
 * counterpart to this call; it is an addition of this library.
 *   Same arguments, results and constraints as sk_gemm_rmsnorm_nvfp4, less
 *   workspace/workspace_bytes, plus m * n <= SK_STATIC_SCRATCH_BYTES / 2:
 *   larger shapes are rejected with SK_ERR_INVALID_ARG before any launch.
 *   The GEMM output goes to a fixed array in the library's device image (one
 *   per device that loads the library, held until the process exits). The
 *   call allocates nothing.
 *   The first call on a device looks up that array's device address (once per
 *   device and CUDA context, with the device current). A device reset destroys
 *   the context that holds the array: the next call looks the address up
 *   again. Every call shares the
 *   array and it keeps the last call's contents; it needs no clearing, since
 *   the GEMM rewrites what the norm then reads. Calls that may run at the same
 *   time on the GPU (unordered streams) race on the array and give wrong
 *   results.
 */
sk_status sk_gemm_rmsnorm_nvfp4_static(const void *x, const void *w, const void *norm_w,
                                       float eps, float gain_center, const float *global_scale,
                                       uint8_t *a, uint8_t *a_sf, void *z_out, int m, int n,
                                       int k, int splits, void *stream);

/*
 * sk_wait_probe -- diagnostic of the bounded-wait path: launches one CTA that
 * waits on an mbarrier that nothing completes, through the same bounded wait
 * the kernels use, for at most limit_us microseconds (1 <= limit_us <=
 * 100000). When the wait runs out the kernel sets SK_DEVICE_WAIT_PROBE in the
 * device status word and returns; the context stays usable. No counterpart
 * on the pages: it tests this library's failure reporting without a fault.
 */
sk_status sk_wait_probe(unsigned limit_us, void *stream);

/*
 * sk_device_status -- HOST-synchronizing diagnostic: copies the library's
 * device status word (an OR of SK_DEVICE_WAIT_* bits set by kernels whose
 * bounded waits ran out) of the current device into *out (host pointer) and,
 * if clear != 0, resets it to 0. Synchronizes the device.
 */
sk_status sk_device_status(uint32_t *out, int clear);

/*
 * sk_convert_probe -- runs one of the device's format conversions used by the
 * NVFP4 epilogue over n FP32 inputs (device pointers), for checking the
 * hardware rounding against a reference:
 *   kind 0: e2m1, out u8 [n]  (code in bits 0..3, round to nearest even, saturating)
 *   kind 1: e4m3fn, out u8 [n] (round to nearest even, saturating to +-448)
 *   kind 2: bf16, out u16 [n] (round to nearest even)
 *   kind 3: e4m3fn byte -> FP32 widening: `in` is read as u8 [n], out FP32 [n]
 */
sk_status sk_convert_probe(int kind, const void *in, void *out, int n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SK_H_ */
