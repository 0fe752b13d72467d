/*
 * gift.h — C ABI of libgift, a GB300 (sm_103a) implementation of GIFT's
 * per-layer gradient codec.
 *
 * GIFT (Geometry-Informed low-precision gradient communication) whitens a weight
 * gradient with the layer's K-FAC input factor before it is quantised to FP8 or
 * NVFP4 for the data-parallel all-reduce, and maps the averaged result back
 * afterwards.  Sources (cited by page title and section):
 *   [notes]    "GIFT 阅读笔记:量化用的坐标系,比量化器本身更重要" (GIFT reading notes,
 *              zhongzhuzhou.org): prerequisites ("What FP8 is", "K-FAC"), core idea
 *              steps 1-3 with eqs. (4)-(14), the three simplifications with eqs.
 *              (15)-(17) and the profiling procedure, Algorithm 1.
 *   [abstract] "GIFT: Geometry-Informed Low-precision Gradient Communication for
 *              LLM Pretraining" (shd-paper.top), abstract: FP8 and NVFP4 formats.
 *
 * Conventions for every entry point
 *   Layout     Matrices are row-major and contiguous.  A gradient W is d_out x d_in
 *              (leading dimension d_in); activations a are T x d_in; delta is T x d_out.
 *   Ownership  The caller owns every buffer: inputs, outputs, factor storage,
 *              workspace (size from gift_workspace_bytes) and the status word.  The
 *              library never allocates device memory and never frees caller memory.
 *              Pointers documented as "device" must point to memory of the device the
 *              context was created for, and that device must be current; pointer
 *              arrays ("host array of device pointers") live in host memory.
 *   Streams    Every call only enqueues work on the caller's stream and returns; no
 *              call synchronises the device.  Results are valid once the stream has
 *              reached the call.
 *   Errors     Two channels.  (1) The return value reports argument validation and
 *              launch failures synchronously (nothing is enqueued on an error other
 *              than GIFT_ERR_CUDA, whose partial work is undefined).  (2) Conditions
 *              only the device can see (a non-finite input, a factor that is not
 *              positive definite, an eigensolver that did not converge) are written
 *              into the caller's device word `d_status` with compare-and-swap from 0:
 *              the first error wins, the library never clears the word.  Pass
 *              d_status = NULL to ignore them.  Outputs are undefined when the word
 *              is non-zero.
 *   Alignment  Any alignment works; 16-byte aligned buffers with d_in a multiple of
 *              4 (FP32) or 16 (codes) take the vectorised paths.
 *   Aliasing   Outputs must not alias inputs unless a parameter says otherwise.
 */
#ifndef GIFT_H_
#define GIFT_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GIFT_VERSION_MAJOR 0
#define GIFT_VERSION_MINOR 1

typedef enum {
  GIFT_OK = 0,
  GIFT_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, workspace too small */
  GIFT_ERR_UNSUPPORTED = 2,   /* valid but not implemented combination                 */
  GIFT_ERR_CUDA = 3,          /* a CUDA launch or runtime call failed                  */
  GIFT_ERR_NONFINITE = 4,     /* device: NaN or Inf in the tensor being scaled         */
  GIFT_ERR_NOT_PD = 5,        /* device: Cholesky pivot <= 0, or sigma/mu <= 0         */
  GIFT_ERR_TIMEOUT = 6,       /* device: a bounded wait gave up                        */
  GIFT_ERR_NOT_CONVERGED = 7  /* device: the eigensolver did not converge              */
} gift_status;

/* Element formats ([notes] prerequisites "What FP8 is"; [abstract] NVFP4).
 *  F32   : no quantisation, codes are the FP32 values (lossless round-trip tests).
 *  E4M3  : 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest finite 448, no Inf.
 *  E5M2  : 1 sign, 5 exponent (bias 15), 2 mantissa bits; largest finite 57344.
 *  NVFP4 : E2M1 codes (largest 6), two per byte with the even column in the low
 *          nibble; one E4M3 scale byte per 16 consecutive elements of a row
 *          (scales[d_out][d_in/16]); one FP32 tensor scale.  Needs d_in % 16 == 0.
 * Rounding is round-to-nearest-even with saturation to the largest finite value;
 * the sign of zero is kept. */
typedef enum { GIFT_FMT_F32 = 0, GIFT_FMT_E4M3 = 1, GIFT_FMT_E5M2 = 2, GIFT_FMT_NVFP4 = 3 } gift_format;

/* Scale groups for FP8 ([notes] "What FP8 is": per tensor or per block).
 *  TENSOR   : one FP32 scale, scales[1].
 *  BLOCK128 : one FP32 scale per 128 x 128 tile, scales[ceil(d_out/128)][ceil(d_in/128)],
 *             edge tiles clipped.
 *  BLOCK512 : one FP32 scale per 512 consecutive elements of the row-major tensor,
 *             scales[ceil(d_out*d_in/512)], the last group shorter (the per-block Euclidean
 *             baseline of the experiments, [notes] three simplifications: block size 512).
 *             Identity and Cholesky transforms only (a rank-r factor returns
 *             GIFT_ERR_UNSUPPORTED).
 * NVFP4 ignores this (its groups are fixed); F32 has no scales. */
typedef enum { GIFT_SCALE_TENSOR = 0, GIFT_SCALE_BLOCK128 = 1, GIFT_SCALE_BLOCK512 = 2 } gift_scaling;

/* Coordinate transforms ([notes] core idea eqs. (11), (14); simplification 1 eq. (16);
 * simplification 2 eq. (17)).
 *  IDENTITY        : the Euclidean path, W~ = W.
 *  LOWRANK         : W~ = W T_A, T_A = sigma^-1/2 I + U (diag(mu^-1/2) - sigma^-1/2) U^T,
 *                    A ~ U diag(mu - sigma) U^T + sigma I with mu the top `rank`
 *                    eigenvalues of A; decode applies T_A^-1.
 *  CHOL_INPUT      : W~ = W L_A^-T, decode W^ = X L_A^T.
 *  CHOL_TWO_SIDED  : W~ = L_G^-1 W L_A^-T, decode W^ = L_G X L_A^T. */
typedef enum {
  GIFT_XF_IDENTITY = 0,
  GIFT_XF_LOWRANK = 1,
  GIFT_XF_CHOL_INPUT = 2,
  GIFT_XF_CHOL_TWO_SIDED = 3
} gift_xform;

/* Arithmetic of the transforms.  FP32: results within FP32 rounding, the transformed and
 * decoded tensors within 1e-5 (relative Frobenius) of exact.  Where the rank-r product runs on
 * the tensor cores (rank-r transforms with d_in % 32 == 0 and 16-byte aligned tensors), FP32
 * splits Pc and U exactly into three BF16 terms and sums the six products with i + j <= 4
 * (what is dropped is below 2^-23 of each |Pc_k U_k|).  TC: two terms and three products
 * (below 2^-15), the transformed tensor within 2e-2; other transforms run the FP32 path. */
typedef enum { GIFT_PREC_FP32 = 0, GIFT_PREC_TC = 1 } gift_precision;

/* Element type of activation inputs. */
typedef enum { GIFT_DT_F32 = 0, GIFT_DT_BF16 = 1 } gift_dtype;

/* One layer's factor: every pointer is device memory owned by the caller.
 *  LOWRANK        : U (d_in x rank, row-major, orthonormal columns), mu (rank values,
 *                   descending, the top eigenvalues of A), sigma (1 value).  planes
 *                   (optional, gift_factor_planes_bytes(d_in) bytes, 16-byte aligned): the
 *                   BF16 term planes of U that the tensor-core kernels read.  When set, the
 *                   codec reads them instead of rebuilding them on every call; they must
 *                   then match U: gift_factor_update refreshes them with U, and
 *                   gift_factor_prepare rebuilds them after the caller changes U.
 *  CHOL_INPUT     : LA and LAinv (d_in x d_in, lower triangular, upper part zero).
 *  CHOL_TWO_SIDED : as CHOL_INPUT plus LG and LGinv (d_out x d_out).
 * Unused pointers may be NULL.  1 <= rank <= 32 and rank <= d_in. */
typedef struct {
  gift_xform kind;
  int d_in, d_out, rank;
  float *U;
  float *mu;
  float *sigma;
  float *LA, *LAinv;
  float *LG, *LGinv;
  void *planes;
} gift_factor;

/* Opaque host context: device properties and tuning; holds no device memory and no
 * per-call state, so calls on different streams may run concurrently. */
typedef struct gift_ctx gift_ctx;

/* Operations for gift_workspace_bytes. */
typedef enum {
  GIFT_OP_FACTOR_UPDATE = 0,
  GIFT_OP_ENCODE = 1,
  GIFT_OP_DECODE = 2,
  GIFT_OP_AMAX = 3,
  GIFT_OP_KFAC_FACTOR = 4,
  GIFT_OP_REDUCE_DECODE = 5
} gift_op;

/* Tunables for gift_set_option. */
typedef enum {
  GIFT_OPT_SUBSPACE_ITERS = 0, /* most power iterations of the rank-r sketch (default 16, 1..64);
                                  they stop earlier once the top Ritz pairs have converged */
  GIFT_OPT_SKETCH = 2,         /* rank-r refresh: 0 (default) forms A Q as a^T (a Q) / T from the
                                  activations and never forms A; 1 forms A = a^T a / T (the
                                  K-FAC product) and multiplies it.  Set it before
                                  gift_workspace_bytes: the two need different workspaces. */
  GIFT_OPT_BARRIER_WAIT = 1,   /* SM clock cycles a CTA of the shared-scale encode waits at its
                                  grid-wide barrier before it gives up, writes GIFT_ERR_TIMEOUT
                                  to d_status and stores no codes (default 2e9, about a second;
                                  0..2e10).  A small value makes the wait run out on purpose: the
                                  kernel still ends and the context stays usable. */
  GIFT_OPT_SMS = 3             /* SMs the context's launches size their grids for (default and
                                  maximum: the device's SM count).  With a fraction of the SMs per
                                  context, calls on several streams run side by side on disjoint
                                  shares of the GPU, which pays for latency-bound calls such as
                                  one layer's decode.  Workspace sizes depend on it: set it
                                  before gift_workspace_bytes. */
} gift_option;

/* Create a context for CUDA device `device` (queries its SM count).  Returns
 * GIFT_ERR_INVALID_ARG for a NULL ctx, GIFT_ERR_CUDA when the device cannot be queried. */
gift_status gift_create(gift_ctx **ctx, int device);
void gift_destroy(gift_ctx *ctx);
gift_status gift_set_option(gift_ctx *ctx, gift_option opt, long long value);
const char *gift_status_string(gift_status s);
int gift_version(void); /* major * 1000 + minor */
/* Text of the last CUDA runtime error that made a libgift call on this thread return
 * GIFT_ERR_CUDA ("no CUDA error" if none); valid until the next failing call. */
const char *gift_last_error(void);

/* Bytes of caller-provided device workspace an operation needs (0 if none).
 * Host-only; returns (size_t)-1 for invalid arguments.  T is used by
 * GIFT_OP_FACTOR_UPDATE and GIFT_OP_KFAC_FACTOR only (the latter also reads d_in = d and
 * ignores kind, format and scaling), rank by the LOWRANK kind only. */
size_t gift_workspace_bytes(const gift_ctx *ctx, gift_op op, gift_xform kind, gift_format fmt,
                            gift_scaling scaling, int d_out, int d_in, int T, int rank);

/* Sizes of one encoded tensor: code bytes, and the number of scale entries (FP32 entries
 * for E4M3/E5M2, E4M3 bytes for NVFP4, 0 for F32).  Host-only. */
gift_status gift_code_sizes(gift_format fmt, gift_scaling scaling, int d_out, int d_in,
                            size_t *code_bytes, size_t *scale_count);

/* Factor refresh ([notes] eq. (4): A = E[a a^T] ~ a^T a / T; core idea step 2 eq. (7):
 * Cholesky; simplification 2 eq. (17): rank-r eigen approximation; Algorithm 1 refreshes
 * it every K steps).
 *  a      : device, T x d_in activations of type a_dt.
 *  delta  : device, T x d_out output gradients of type d_dt (CHOL_TWO_SIDED only, else NULL).
 *  f      : f->kind selects the factor; its buffers receive the result.
 *  LOWRANK: randomised block subspace iteration on A with a seeded Gaussian start of
 *           k = min(64, d_in) columns (Philox4x32-10 from `seed`).  For d_in > 64 it runs
 *           in FP32 with every product on the tensor cores (FP32 operands split exactly
 *           into BF16 terms, one fresh FP32 accumulator per 64-deep chunk): each power step
 *           forms Y = A Q (by default as a^T (a Q) / T, A never formed; GIFT_OPT_SKETCH
 *           selects the explicit product) and re-orthonormalises Q by CholQR2 with
 *           compensated FP32 Gram sums; Rayleigh-Ritz steps (FP32 one-sided Jacobi) rotate
 *           Q on the first two steps and every fourth, and stop the iteration once each of
 *           the top `rank` Ritz pairs has a residual ||A u - theta u|| <= 1e-4 theta (at
 *           most GIFT_OPT_SUBSPACE_ITERS steps, default 16).  The last Rayleigh-Ritz step takes
 *           Q^T A Q as the Gram matrix of a Q.  For d_in <= 64 the Gram, Cholesky and
 *           eigensolve run in FP64 on A itself.  U = Q V[:, :rank]; sigma =
 *           (tr A - sum mu) / (d_in - rank) (sigma = 1 when rank == d_in).  d_status:
 *           NOT_PD when sigma or a mu is <= 0, NOT_CONVERGED when the final Jacobi sweeps do
 *           not converge.
 *  CHOL_* : A (and G) are formed in FP32 and factored in FP64; L and L^-1 are stored in
 *           FP32.  d_status: NOT_PD on a non-positive pivot.
 *  prec   : GIFT_PREC_FP32 forms A (and G) on the tensor cores from exact three-term BF16
 *           splits of FP32 activations (BF16 activations are their own single term), each
 *           64-deep chunk in a fresh FP32 accumulator: FP32 accuracy.  GIFT_PREC_TC with BF16
 *           activations (d a multiple of 256, T of 64) accumulates over all of T inside the
 *           tensor cores (their summation order, not round to nearest), and the rank-r
 *           sketch keeps two terms of its FP32 operands (about 16 mantissa bits).
 *  ws     : device workspace of gift_workspace_bytes(GIFT_OP_FACTOR_UPDATE, ..., T, ...)
 *           bytes (term planes of the activations and of Q, the partial sums, the FP64
 *           Cholesky scratch).
 * LOWRANK with d_in > 64 allocates nothing, never waits on the host and enqueues the same
 * launches on every call (once the Ritz residuals converge, the remaining launches return at
 * once), so the call can be captured into a CUDA graph and replayed; a replay gives the eager
 * call's factor bit for bit.
 * Returns INVALID_ARG on null pointers, T < 1, rank outside [1, min(32, d_in)]. */
gift_status gift_factor_update(gift_ctx *ctx, gift_factor *f, const void *a, gift_dtype a_dt, int T,
                               const void *delta, gift_dtype d_dt, uint64_t seed, gift_precision prec,
                               void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream);

/* The factor refresh from K-FAC factors the caller already holds: gift_factor_update
 * without its first step, for factors combined before they are factored (the average of A
 * over the data-parallel replicas, or a running average across refreshes, both of which
 * gift_kfac_factor's output can feed).  [notes] eq. (4) defines A; the factoring is the same
 * as gift_factor_update's (core idea step 2 eq. (7), simplification 2 eq. (17)), except that
 * the rank-r sketch multiplies A explicitly and its last Rayleigh-Ritz step forms Q^T (A Q).
 *  A  : device, d_in x d_in FP32, row-major, symmetric positive semi-definite; read only.
 *  G  : device, d_out x d_out FP32 (CHOL_TWO_SIDED only, else NULL); read only.
 *  ws : gift_workspace_bytes(GIFT_OP_FACTOR_UPDATE, ..., T = 0, ...) bytes.
 * Returns INVALID_ARG on a null A (or G for CHOL_TWO_SIDED) and on the cases
 * gift_factor_update rejects; d_status as for gift_factor_update. */
gift_status gift_factor_update_from_kfac(gift_ctx *ctx, gift_factor *f, const float *A, const float *G,
                                         uint64_t seed, gift_precision prec, void *ws, size_t ws_bytes,
                                         int *d_status, cudaStream_t stream);

/* Bytes of the optional U term planes of a rank-r factor (gift_factor.planes). */
size_t gift_factor_planes_bytes(int d_in);

/* Rebuild f->planes from f->U (LOWRANK, planes set); asynchronous on `stream`.  Returns
 * INVALID_ARG when the factor is not LOWRANK or has no U or planes. */
gift_status gift_factor_prepare(gift_ctx *ctx, const gift_factor *f, cudaStream_t stream);

/* The K-FAC factor alone ([notes] prerequisites, eq. (4): A = a^T a / T), the first step of
 * gift_factor_update, for callers that combine factors before factoring them (for example
 * averaging A over the data-parallel replicas or across refreshes).
 *  a     : device, T x d activations of type a_dt, row-major.
 *  prec  : as in gift_factor_update; without a workspace (GIFT_PREC_FP32 only) the sums
 *          run in FP32 SIMT arithmetic.
 *  A_out : device, d x d FP32, row-major; receives the full symmetric matrix.
 *  ws    : device workspace of gift_workspace_bytes(GIFT_OP_KFAC_FACTOR, ..., d_out, d_in = d,
 *          T, ...) bytes (the activations' BF16 transpose or term planes); may be NULL with
 *          GIFT_PREC_FP32.
 * Returns INVALID_ARG on null pointers, d < 1, T < 1, or a workspace too small for TC. */
gift_status gift_kfac_factor(gift_ctx *ctx, const void *a, gift_dtype a_dt, int T, int d, gift_precision prec,
                             float *A_out, void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream);

/* Amax of the tensor that gift_encode would quantise (the transformed gradient, plus the
 * residual when one is given), max-accumulated into amax_accum: the AllReduceMax of the
 * scale in Algorithm 1, modelled on one GPU by calling this once per replica on one
 * accumulator the caller set to 0 beforehand.  amax_accum holds 1 float (TENSOR, NVFP4)
 * or ceil(d_out/128) x ceil(d_in/128) floats (BLOCK128).  d_status: NONFINITE. */
gift_status gift_amax(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in,
                      gift_format fmt, gift_scaling scaling, gift_precision prec,
                      const float *residual, float *amax_accum, void *ws, size_t ws_bytes,
                      int *d_status, cudaStream_t stream);

/* Encode one gradient ([notes] Algorithm 1: whiten, add the error-feedback residual,
 * Scale, Q; eq. (13) CommFP8 input side).
 *  f         : NULL or kind IDENTITY for the Euclidean path.
 *  W         : device, d_out x d_in FP32 gradient.
 *  amax_in   : device, nullable.  When given, the scale uses this amax (shared scale of the
 *              Euclidean path) instead of the tensor's own: 1 float (TENSOR, NVFP4) or one
 *              per 128 x 128 block.
 *  residual  : device, nullable, d_out x d_in FP32 error-feedback buffer R in whitened
 *              coordinates: U~ = W~ + R is quantised, then R <- U~ - Dequantize(Q(U~)).
 *  codes     : device, gift_code_sizes bytes (F32: d_out*d_in floats).
 *  scales    : device, gift_code_sizes entries (FP32, or E4M3 bytes for NVFP4).
 *  tensor_scale : device, 1 float, NVFP4 only (else NULL).
 *  transformed_out : device, nullable, receives U~ in FP32 (parity and fidelity checks).
 *  amax_out  : device, nullable, receives the amax used (same shape as amax_in).
 *  Scale rule: s = amax / FMAX stored, elements scaled by m = FMAX / amax (two FP32
 *  divisions, FMAX = 448 or 57344); amax = 0 gives s = m = 0; m beyond FP32 is clamped.
 *  NVFP4: s_t = amax / 2688; per group of 16, e = E4M3(group_amax / (6 s_t)),
 *  r = 1 / (e s_t), code = E2M1(x r).
 *  d_status: NONFINITE when the tensor holds NaN/Inf.  W must not alias codes or
 *  residual. */
gift_status gift_encode(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in,
                        gift_format fmt, gift_scaling scaling, gift_precision prec,
                        const float *amax_in, float *residual, void *codes, void *scales,
                        float *tensor_scale, float *transformed_out, float *amax_out,
                        void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream);

/* Encode the R data-parallel replicas of one layer's gradient, which share the factor f
 * ([notes] Algorithm 1, the per-worker encode before AllReduceSum, for R workers modelled on
 * one GPU).  The result is identical to R gift_encode calls with the same arguments (and
 * no residual or transformed_out); on the rank-r path with per-tensor FP8 or NVFP4 scaling
 * each group of up to 8 replicas is encoded by three launches (projection of every replica,
 * Pc, then apply and pack), which overlap the read of one replica's gradient with the pack
 * of the previous one.
 *  W, codes, scales, tensor_scales, amax_in, amax_out : host arrays of R device pointers,
 *              each element as in gift_encode; amax_in and amax_out may be NULL (no
 *              caller amax / no copy for any replica), tensor_scales may be NULL unless
 *              fmt is NVFP4, scales may be NULL for F32.
 *  ws        : one gift_workspace_bytes(GIFT_OP_ENCODE, ...) workspace, used by all replicas
 *              in stream order.  1 <= R <= 64.  Every replica's arguments are checked
 *              before anything is enqueued.  d_status: as gift_encode. */
gift_status gift_encode_replicas(gift_ctx *ctx, const gift_factor *f, int R, const float *const *W,
                                 int d_out, int d_in, gift_format fmt, gift_scaling scaling,
                                 gift_precision prec, const float *const *amax_in,
                                 void *const *codes, void *const *scales,
                                 float *const *tensor_scales, float *const *amax_out, void *ws,
                                 size_t ws_bytes, int *d_status, cudaStream_t stream);

/* Encode R replicas with one shared scale: the amax is the max over the replicas of the amax
 * each would use on its own (the AllReduceMax of the scale in [notes] Algorithm 1, which the
 * Euclidean baseline applies on every step), and every replica is packed with it.  The result
 * is identical to zeroing a word, gift_amax_replicas into it, then gift_encode_replicas with
 * that word as every replica's amax_in.  The identity transform with per-tensor FP8 scaling
 * (16-byte aligned gradients, d_out*d_in a multiple of 4, 4-byte aligned codes) is one
 * cooperative launch: the amax of every replica, a grid-wide barrier, then the pack with the
 * replicas taken last to first, so that it reads first what the amax pass read last (L2 still
 * holds up to ~100 MB of it).  Other kinds and formats take the amax launch(es), then the
 * encode launches of gift_encode_replicas.
 *  W, codes, scales, tensor_scales : host arrays of R device pointers, each element as in
 *              gift_encode (tensor_scales only for NVFP4, may be NULL otherwise).
 *  shared_amax_out : device, 1 float, nullable: the shared amax.
 *  ws        : gift_workspace_bytes(GIFT_OP_ENCODE, ...).  1 <= R <= 64.
 * Errors: INVALID_ARG for F32 (no scale) and for block-128 FP8 scaling (the scales are per
 * block: nothing to share), and for any replica's invalid arguments, before anything is
 * enqueued.  d_status: NONFINITE; TIMEOUT when the grid-wide barrier wait (bounded at about a
 * second) gives up, in which case the codes are not written. */
gift_status gift_encode_replicas_shared(gift_ctx *ctx, const gift_factor *f, int R,
                                        const float *const *W, int d_out, int d_in,
                                        gift_format fmt, gift_scaling scaling,
                                        gift_precision prec, void *const *codes,
                                        void *const *scales, float *const *tensor_scales,
                                        float *shared_amax_out, void *ws, size_t ws_bytes,
                                        int *d_status, cudaStream_t stream);

/* The shared amax of R replicas (the AllReduceMax of the scale in [notes] Algorithm 1, for R
 * workers modelled on one GPU): max-accumulates into amax_accum the amax that gift_amax would
 * give for each of the R tensors W[r] (host array of R device pointers, 1 <= R <= 64).  Same
 * result as R gift_amax calls without residual; identity and rank-r factors with per-tensor
 * scaling take one streaming pass over all replicas.  ws: gift_workspace_bytes(GIFT_OP_AMAX,
 * ...).  d_status: NONFINITE. */
gift_status gift_amax_replicas(gift_ctx *ctx, const gift_factor *f, int R, const float *const *W,
                               int d_out, int d_in, gift_format fmt, gift_scaling scaling,
                               gift_precision prec, float *amax_accum, void *ws, size_t ws_bytes,
                               int *d_status, cudaStream_t stream);

/* Replica reduce: out = (sum_r deq_r) / R in FP32, adding replicas in order r = 0..R-1
 * with each replica dequantised with its own scale ([notes] eq. (1) data-parallel average;
 * Algorithm 1 AllReduceSum, Dequantize, divide by N — modelled on one GPU over R code
 * buffers held in this GPU's memory).
 *  codes, scales, tensor_scales : host arrays of R device pointers (tensor_scales only for
 *                                 NVFP4, may be NULL otherwise; scales NULL for F32).
 *  avg_out : device, d_out x d_in FP32.  1 <= R <= 64. */
gift_status gift_replica_reduce(gift_ctx *ctx, int R, const void *const *codes,
                                const void *const *scales, const float *const *tensor_scales,
                                gift_format fmt, gift_scaling scaling, int d_out, int d_in,
                                float *avg_out, int *d_status, cudaStream_t stream);

/* Decode: dequantise (when `in` holds codes) and map back to the gradient's coordinates
 * ([notes] eq. (14); Algorithm 1 multiplies by L_A^T).
 *  in         : device; codes of `fmt` when in_is_codes != 0 (with scales / tensor_scale as
 *               written by gift_encode), else a d_out x d_in FP32 tensor in whitened
 *               coordinates (for example gift_replica_reduce's output).
 *  W_out      : device, d_out x d_in FP32.  Must not alias `in`.
 *  ws         : gift_workspace_bytes(GIFT_OP_DECODE, ...) bytes. */
gift_status gift_decode(gift_ctx *ctx, const gift_factor *f, const void *in, int in_is_codes,
                        const void *scales, const float *tensor_scale, gift_format fmt,
                        gift_scaling scaling, gift_precision prec, int d_out, int d_in, float *W_out,
                        void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream);

/* Replica reduce and decode in one call ([notes] Algorithm 1: AllReduceSum, Dequantize,
 * divide by N, then map back with the factor, eq. (14)): W_out = decode(average of the R
 * replicas' codes).  It enqueues gift_replica_reduce into avg_out (or into the workspace) and
 * then gift_decode of that average, back to back, so that the decode reads the average from
 * L2; the results are those two calls' (the average bit for bit).
 *  codes, scales, tensor_scales : as gift_replica_reduce.
 *  avg_out : device, nullable, d_out x d_in FP32: receives the average.
 *  W_out   : device, d_out x d_in FP32.  Must alias neither the codes nor avg_out.
 *  ws      : gift_workspace_bytes(GIFT_OP_REDUCE_DECODE, ...) bytes.  1 <= R <= 64. */
gift_status gift_reduce_decode(gift_ctx *ctx, const gift_factor *f, int R, const void *const *codes,
                               const void *const *scales, const float *const *tensor_scales, gift_format fmt,
                               gift_scaling scaling, gift_precision prec, int d_out, int d_in, float *avg_out,
                               float *W_out, void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream);

/* Boundary-hit profiler ([notes] simplification 3: encode the flattened gradient with the
 * scale that would be used and count codes on the upper or lower boundary of the FP8
 * format).  Euclidean encode with the tensor's own scale (per tensor or per block);
 * adds into d_counts[0] the number of codes whose magnitude is the largest finite code,
 * into d_counts[1] the number of non-zero elements whose code is zero, and into
 * d_counts[2] the number of elements.  Counts accumulate across calls (a profiling
 * window); the caller zeroes them.  fmt: E4M3 or E5M2.
 *  ws : gift_workspace_bytes(GIFT_OP_AMAX, IDENTITY, ...) bytes (one amax word).
 *  d_status: NONFINITE. */
gift_status gift_boundary_hit_rate(gift_ctx *ctx, const float *W, int d_out, int d_in,
                                   gift_format fmt, gift_scaling scaling,
                                   unsigned long long *d_counts, void *ws, size_t ws_bytes,
                                   int *d_status, cudaStream_t stream);

/* The boundary-hit profiler over several tensors in one call (the profiling window's pass over
 * a model's layers): for each tensor t the counts gift_boundary_hit_rate would add, added into
 * d_counts[3 t .. 3 t + 2].  No counterpart in the pages beyond the per-tensor procedure; it
 * exists so that a model's layers take two launches (every tensor's amax, then every tensor's
 * counts) instead of two or three each.
 *  W, d_out, d_in : host arrays of n_tensors device pointers and shapes (FP32, row-major).
 *  d_counts       : device, n_tensors x 3 unsigned 64-bit, added into.
 *  ws             : gift_workspace_bytes(GIFT_OP_AMAX, IDENTITY, ..., 1, 1, ...) bytes (64
 *                   amax words: tensors are taken 64 at a time); per-tensor calls for the
 *                   block scalings.
 * Returns INVALID_ARG on any null pointer or shape <= 0 (nothing enqueued).  d_status:
 * NONFINITE. */
gift_status gift_boundary_hit_rates(gift_ctx *ctx, int n_tensors, const float *const *W, const int *d_out,
                                    const int *d_in, gift_format fmt, gift_scaling scaling,
                                    unsigned long long *d_counts, void *ws, size_t ws_bytes, int *d_status,
                                    cudaStream_t stream);

/* Fragile-layer selection after a profiling window ([notes] simplification 3: boundary-hit
 * rates averaged over the profiling window, upper and lower rates summed into a fragility
 * score; the geometry-aware branch goes to the layers before the clear drop in that score).
 * Host only (no context, no device).
 *  L       : number of layers, >= 1.
 *  counts  : host, L x 3 unsigned 64-bit: layer l's (upper, lower, n) summed over the window,
 *            as gift_boundary_hit_rate accumulates them.  n is the layer's element count at
 *            each step times the steps, so upper + lower over n is the window mean of the
 *            per-step rate.  upper <= n and lower <= n, else INVALID_ARG.
 *  k       : > 0: select the k highest-scoring layers.  0: select at the knee, the k in
 *            [k_min, min(k_max, L - 1)] with the largest drop between consecutive ranked
 *            scores (equal drops: the smaller k); with k_min = L, all L.
 *            1 <= k_min <= k_max <= L is required when k = 0; otherwise both are ignored.
 *  order   : host, L ints out: layer indices by descending score, ties to the lower index.
 *            The selected layers are order[0 .. *k_out).
 *  scores  : host, L doubles out (nullable): (upper + lower) / n per layer in double,
 *            0 when n = 0.
 *  k_out   : host, 1 int out.
 * Errors (INVALID_ARG, nothing written): L < 1, null counts/order/k_out, k outside [0, L],
 * a bad k_min/k_max with k = 0, counts above n. */
gift_status gift_select_fragile(int L, const unsigned long long *counts, int k, int k_min, int k_max,
                                int *order, double *scores, int *k_out);

/* Rank-r encode that allocates nothing (the paper has no counterpart; this is a library
 * convenience).  Same result as gift_encode with a LOWRANK factor, GIFT_PREC_FP32, E4M3 or
 * E5M2 and per-tensor scaling, but without a caller workspace: for callers that cannot allocate
 * device memory at the point where they encode, such as code running inside a gradient or
 * communication hook while the framework's allocator must not grow, or C programs with no
 * allocator of their own.  Its scratch (about 17 MiB) is a fixed array inside the library,
 * present on every GPU that loads it until the process exits.
 *  Limits: d_out <= 4096, d_in <= 16384, and the split-K projection partials must fit the scratch
 *  (ceil-split count x d_out x 32 floats <= 2^21); beyond them the call returns
 *  GIFT_ERR_INVALID_ARG and enqueues nothing.
 *  Set-up: the first call on a device (with that device current) looks up the array's
 *  device address; make that first call before any stream capture begins.
 *  Concurrency: all calls on a device share the scratch; calls whose GPU work overlaps
 *  (unordered streams) race on it.  Order them on one stream or with events.
 *  amax_in, amax_out, d_status may be NULL; scales receives one FP32 value. */
gift_status gift_encode_lowrank_noalloc(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in,
                                        gift_format fmt, const float *amax_in, void *codes, float *scales,
                                        float *amax_out, int *d_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GIFT_H_ */
