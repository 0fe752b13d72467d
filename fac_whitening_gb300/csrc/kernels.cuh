// Internal launcher declarations of libgift (host side of each kernel file).
#pragma once

#include "common.cuh"

// Host context behind the opaque gift_ctx handle.
struct gift_ctx {
  int device;
  int device_sms;           // SMs of the device
  int sms;                  // SMs this context's launches size their grids for (<= device_sms)
  int subspace_iters;
  long long barrier_wait;   // clock cycles a CTA waits at a streaming grid barrier
  int sketch;               // rank-r refresh: 0 implicit a^T (a Q) / T, 1 explicit A Q
};

namespace gift {

constexpr long long kDefaultBarrierWait = 2000000000LL;   // clock cycles, about a second

struct Launch {
  cudaStream_t stream;
  int sms;       // streaming multiprocessors of the device
  int *status;   // caller's device status word (nullable)
  long long barrier_wait = kDefaultBarrierWait;   // bounded wait of the streaming grid barriers
};

struct ReduceArgs {
  const void *codes[kMaxReplicas];
  const void *scales[kMaxReplicas];
  const float *tscales[kMaxReplicas];
};

// Several tensors of one size in one streaming launch (quant.cu).
struct MultiArgs {
  const float *x[kMaxReplicas];
  uint8_t *codes[kMaxReplicas];        // pack: E4M3 / E5M2 codes of each tensor
  float *scale[kMaxReplicas];          // pack: each tensor's scale s
  const float *amax_in[kMaxReplicas];  // pack: the amax each tensor is scaled with
  float *amax_out[kMaxReplicas];       // pack: nullable copies of it
  uint32_t *amax_bits[kMaxReplicas];   // amax: max-accumulated |x| bit pattern of each tensor
};

// Tensors of any sizes for one multi-tensor launch (the profiler's batched hit counts).
struct HitsArgs {
  const float *x[kMaxReplicas];
  size_t n[kMaxReplicas];
};

// ---- quant.cu ---------------------------------------------------------------------------
// amax words zeroed, every tensor's amax, then every tensor's hits added into counts[3 t ..]
cudaError_t launch_hits_multi(const Launch &L, int fmt, const HitsArgs &a, int T, uint32_t *amax_bits,
                              unsigned long long *counts);
cudaError_t launch_amax(const Launch &L, const float *x, const float *r, size_t n, float *amax_accum);
cudaError_t launch_pack_tensor(const Launch &L, int fmt, const float *x, float *r, size_t n, const float *amax,
                               uint8_t *codes, float *scale, float *amax_out, float *tout);
cudaError_t launch_pack_f32(const Launch &L, const float *x, float *r, size_t n, float *out, float *tout);
// mode 0: pack, 1: amax only (max-accumulated into amax_out), 2: count boundary hits
cudaError_t launch_block128(const Launch &L, int fmt, int mode, const float *x, float *r, int d_out, int d_in,
                            const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                            unsigned long long *counts);
// 1-D blocks of 512 consecutive elements; modes as launch_block128 (amax_out of mode 1 is
// max-accumulated per block)
cudaError_t launch_block512(const Launch &L, int fmt, int mode, const float *x, float *r, size_t n,
                            const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                            unsigned long long *counts);
cudaError_t launch_pack_nvfp4(const Launch &L, const float *x, float *r, size_t n, const float *amax,
                              uint8_t *codes, uint8_t *bscale, float *tscale, float *amax_out, float *tout);
cudaError_t launch_hits_tensor(const Launch &L, int fmt, const float *x, size_t n, const float *amax,
                               unsigned long long *counts);
cudaError_t launch_reduce(const Launch &L, const ReduceArgs &a, int R, int fmt, int scaling, int d_out, int d_in,
                          float *out);
// 16-byte aligned tensors, n a multiple of 4 (and 4-byte aligned codes for the pack).
bool multi_ok(const MultiArgs &a, int R, size_t n, bool pack);
cudaError_t launch_amax_multi(const Launch &L, const MultiArgs &a, int R, size_t n);
cudaError_t launch_pack_tensor_multi(const Launch &L, int fmt, const MultiArgs &a, int R, size_t n);
// the R tensors of a (x, codes, scale, amax_out) packed with the max of their amax (cooperative
// launch); ws: two words, zero before the launch; shared_out nullable
cudaError_t launch_encode_shared(const Launch &L, int fmt, const MultiArgs &a, int R, size_t n, uint32_t *ws,
                                 float *shared_out);

// ---- lowrank.cu -------------------------------------------------------------------------
// Split-K projection P = X U (d_out x 32, zero-padded beyond rank); partials to `part`.
int lr_proj_splits(int sms, int d_out, int d_in);
cudaError_t launch_lr_proj(const Launch &L, const float *X, int d_out, int d_in, const float *U, int rank,
                           float *part, int nsplit);
// Pc[row][k] = c_k * sum_s part[s][row][k]; c from (mu, sigma), inverse = map-back coefficients.
// pc_terms (nullable): also the BF16 term planes of Pc for the tensor-core apply.
cudaError_t launch_lr_finalize(const Launch &L, const float *part, int nsplit, int d_out, const float *mu,
                               const float *sigma, int rank, bool inverse, float *Pc, float *pc_terms = nullptr,
                               int terms = 3);
// Everything the apply needs before it runs: P = X U, Pc and, when `split` is given and the
// shape allows, the tensor-core operand planes (tensor-core projection where eligible,
// otherwise the FP32-SIMT projection and finalize).  `part` holds lr_part_floats floats.
cudaError_t lr_prepare_all(const Launch &L, const float *U, const float *mu, const float *sigma, int rank,
                           const float *X, int d_out, int d_in, bool inverse, bool tc_precision, float *part,
                           float *Pc, float *split, const void *cached_planes = nullptr);
size_t lr_part_floats(int sms, int d_out, int d_in);
// Fused apply V = alpha X + Pc U^T (+ R), alpha = sigma^-1/2 (or sigma^1/2 for the map back).
enum LrEpi { LR_AMAX = 0, LR_PACK_TENSOR = 1, LR_BLOCK = 2, LR_NVFP4 = 3, LR_STORE = 4, LR_BLOCK_AMAX = 5 };
struct LrApply {
  const float *X;
  const float *U;
  const float *Pc;
  const float *sigma;
  int rank, d_out, d_in;
  bool inverse;
  float *R;                 // residual (nullable)
  float *tout;              // transformed copy (nullable)
  const float *amax_in;     // shared amax (nullable)
  float *amax_ws;           // LR_AMAX / LR_BLOCK_AMAX: max-accumulated; LR_PACK_TENSOR / NVFP4: read
  uint8_t *codes;
  void *scales;
  float *tscale;
  float *amax_out;
  float *out;               // LR_STORE
  int terms;                // tensor-core path: 1 = TC precision (two BF16 terms, three products),
                            // otherwise FP32 precision (three BF16 terms, six products)
  float *split;             // BF16 term planes (tc.cuh): Pc planes (2 x d_out x 32 floats), then U
  unsigned int *grid_counter;   // fused encode: grid-barrier word, zero before the launch
  const uint16_t *u_planes;     // U term planes for the apply (2 x d_in rows of 64 BF16)
  const uint16_t *ut_planes;    // U^T term planes for the projection (3 x 32 rows of d_in BF16)
};
cudaError_t launch_lr_apply(const Launch &L, int epi, int fmt, const LrApply &a);
// lowrank_tc.cu: the same apply on tcgen05 tensor cores (vectorised shapes only)
bool lr_apply_tc_ok(const LrApply &a, int epi);
size_t lr_pipe_split_floats(int d_out, int d_in);
cudaError_t launch_lr_split_u(const Launch &L, const LrApply &a);
cudaError_t launch_lr_apply_tc(const Launch &L, int epi, int fmt, const LrApply &a, bool single_term);
// Fused encode (transform, grid-wide amax, pack; W read once) for per-tensor FP8 and NVFP4
// on shapes whose tiles fit in tensor memory across the SMs; cooperative launch.
bool lr_encode_fused_ok(const Launch &L, const LrApply &a, int epi);
cudaError_t launch_lr_encode_fused(const Launch &L, int epi, int fmt, const LrApply &a);
// One tensor of a batched rank-r encode (tensors that share the factor and the shape).
struct LrEncodeItem {
  const float *X;
  uint8_t *codes;
  void *scales;
  float *tscale, *amax_out, *tout;
  const float *amax_in;
};
constexpr int kEncodeBatchMax = 16;   // tensors per batched launch; the amax words precede the
                                      // grid-barrier word (at index kEncodeBatchMax)
// Tensors per batched launch that the codec workspace holds partials for.
constexpr int kBatchWs = 8;
// lowrank_batch.cu: the rank-r encode of up to kEncodeBatchMax tensors sharing a factor, in
// two streaming passes (projection of every tensor, then apply, tensor amax and pack with the
// tensor in tensor memory).  Needs the U planes (a.u_planes, a.ut_planes), a.amax_ws[0..nb)
// zeroed for the tensors without a caller amax, a.grid_counter zeroed; part holds nb x
// lr_batch_part_floats floats and pc_planes nb x 2 x d_out rows of 64 BF16.
int lr_batch_plan(int sms, int d_out, int d_in, int *cpr_out);
size_t lr_batch_part_floats(int sms, int d_out, int d_in);
bool lr_encode_batch_ok(const Launch &L, const LrApply &a, int epi);
cudaError_t launch_lr_encode_batch(const Launch &L, int epi, int fmt, const LrApply &a, const float *mu,
                                   float *part, uint16_t *pc_planes, int nb, const LrEncodeItem *items);
// lowrank_proj_tc.cu: the projection and the finalize on the tensor cores.  The tensor-core
// workspace ("split", lr_pipe_split_floats floats) holds, in order: the Pc term planes
// (2 x d_out rows of 64 BF16), the U term planes for the apply (2 x d_in rows), the U^T term
// planes for the projection (3 x 32 rows of d_in BF16) and one counter per 128-row block.
struct LrPlanes {
  uint16_t *pc, *u, *ut;
  unsigned int *counters;
  int ncounters;
};
LrPlanes lr_planes(float *split, int d_out, int d_in);
// U planes of a factor: its cached planes (gift_factor.planes, laid out [u | ut]) when given,
// otherwise the workspace's.
void lr_u_planes(const void *cached, float *split, int d_out, int d_in, const uint16_t **u, const uint16_t **ut);
size_t lr_factor_planes_bytes(int d_in);
// Write the U planes of (U, rank) into a factor's cached planes.
cudaError_t launch_lr_factor_planes(const Launch &L, const float *U, int d_in, int rank, void *planes);
int lr_proj_tc_splits(int sms, int d_out, int d_in);
bool lr_proj_tc_ok(const float *X, int d_in, const float *split);
// U planes in both layouts (and the counters zeroed); then P, Pc and the Pc planes.
cudaError_t launch_lr_split_u_all(const Launch &L, const float *U, int d_out, int d_in, int rank, int nplanes_apply,
                                  float *split);
cudaError_t launch_lr_proj_tc(const Launch &L, const float *X, int d_out, int d_in, const float *mu,
                              const float *sigma, int rank, bool inverse, bool tc_precision, float *part, float *Pc,
                              float *split, const uint16_t *ut_planes);

// syrk_tc.cu: A = scale * x^T x for BF16 x (T x d) on tcgen05 (lower tiles; mirror after).
// `at` is scratch of syrk_tc_scratch_bytes(d, T) bytes (the transpose of x).
bool syrk_tc_ok(int d, int T, const void *a, const void *at, const float *out);
size_t syrk_tc_scratch_bytes(int d, int T);
cudaError_t launch_syrk_tc(const Launch &L, const void *a, int T, int d, float scale, void *at, float *out);
// a (T x d BF16, d and T multiples of 64) -> at (d x T)
cudaError_t launch_transpose_bf16(const Launch &L, const void *a, int T, int d, void *at);

// factor_tc.cu: the FP32 pieces of the rank-r refresh (k = 64 sketch columns); every launch
// returns at once while *skip != 0 (skip nullable)
int refresh_gram_ctas(int sms, int d);
// out (k x k) = X^T Y for d x k X and Y; parts holds refresh_gram_ctas x k x k floats
cudaError_t launch_gram_tall(const Launch &L, const float *X, const float *Y, int d, int k, float *parts, float *out,
                             bool sym, const int *skip, float scale = 1.0f);
// tr(a^T a / T) from the activations; part holds nparts doubles (one per CTA)
cudaError_t launch_trace_acts32(const Launch &L, const void *a, bool bf16, int T, int d, double *part, int nparts,
                                double *tr);
// G = L L^T (k = 64); L lower-triangular, upper part zero
cudaError_t launch_chol32(const Launch &L, const float *G, int k, float *Lout, const int *skip);
// at most max_sweeps sweeps; report: NOT_CONVERGED into the status word when they run out
cudaError_t launch_jacobi32(const Launch &L, const float *B, int k, float *evals, float *V, int max_sweeps,
                            bool report, const int *skip);
// out = X L^-T for X d x 64 and L 64 x 64 lower-triangular (out may be X)
cudaError_t launch_right_trsm64(const Launch &L, const float *X, int d, const float *Lm, float *out,
                                const int *skip);
// Y <- Y V in place with the Ritz residuals' partial sums of squares (ritz_rotate_ctas x 64
// floats), then the convergence flag from them
int ritz_rotate_ctas(int sms, int d);
cudaError_t launch_ritz_rotate(const Launch &L, float *Y, const float *Q, int d, const float *V, const float *theta,
                               float *res_parts, const int *skip);
cudaError_t launch_ritz_check(const Launch &L, const float *res_parts, int nparts, const float *theta, int r,
                              int *flag);
cudaError_t launch_trace_diag(const Launch &L, const float *A, int d, double *tr);

// Sets a kernel's opt-in dynamic shared-memory size once per device and kernel (so no
// attribute call happens inside a stream capture after the first eager call).  Keyed on the
// kernel itself: instantiations that share a function type keep separate flags.
template <auto Kernel>
cudaError_t ensure_dynamic_smem(int bytes) {
  static int done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = bytes;
  return e;
}

// Last CUDA error seen by a libgift call on this thread (see gift_last_error).
void record_cuda_error(cudaError_t e);

// ---- linalg.cu --------------------------------------------------------------------------
// C[M x N] = alpha * op(A) op(B), FP32 accumulate.  op(A) = A (M x K, lda) or A^T (A is K x M).
// op(B) = B (K x N, ldb) or B^T (B is N x K).  a_lower: op(A)[m][k] = 0 for k > m;
// b_lower_t: op(B)[k][n] = 0 for k > n.  lower_tiles: only tiles with n0 <= m0 (square tiles).
struct GemmArgs {
  const void *A;
  const void *B;
  float *C;
  int M, N, K, lda, ldb, ldc;
  bool transA, transB;
  bool a_bf16, b_bf16;
  bool a_lower, b_lower_t, lower_tiles;
  float alpha;
};
cudaError_t launch_sgemm(const Launch &L, const GemmArgs &g);
// gemm_tc.cu: the same product on tcgen05 with the operands split exactly into nt BF16 term
// planes (nt = 3: six products, FP32 precision; nt = 2: three products) in ws
// (gemm_tc_ws_bytes(M, N, K, nt) bytes, 16-byte aligned).  FP32 operands, no transA.
bool gemm_tc_ok(const GemmArgs &g, const void *ws);
size_t gemm_tc_ws_bytes(int M, int N, int K, int nterms);
size_t gemm_tc_plane_bytes(int rows, int K, int nterms);
cudaError_t launch_gemm_tc(const Launch &L, const GemmArgs &g, int nt, void *ws);
// The planes alone (rows x K, or the transpose of a K x rows source; rows padded to 128 and K
// to 64 with zeros; blocked: each 128-row x 64-K tile contiguous), and the product of two
// plane sets C = alpha A B^T (M x N, K):
//   nta / ntb   term planes of A and B (1..3; a BF16 source is its own single term);
//   fp32        keep the products x_i y_j with i + j <= 2 (0-based), else i + j <= 1;
//   a_lower / b_lower  row i of A (row j of B) is zero beyond k = i (j);
//   lower_tiles only the 128 x 128 tiles on or below the diagonal (M == N; mirror after);
//   ksplit > 1  K in ksplit slices, partial products in parts (gemm_tc_parts_floats floats),
//               then summed in slice order;
//   skip        nullable device flag: every launch does nothing while it is non-zero.
struct GemmPlanes {
  const uint16_t *pa = nullptr, *pb = nullptr;   // blocked term planes (launch_split_planes)
  int M = 0, N = 0, K = 0;
  int nta = 1, ntb = 1;
  bool fp32 = true;
  bool a_lower = false, b_lower = false, lower_tiles = false;
  int ksplit = 1;
  float *parts = nullptr;
  float alpha = 1.0f;
  float *C = nullptr;
  int ldc = 0;
  const int *skip = nullptr;
};
cudaError_t launch_split_planes(const Launch &L, const float *src, int rows, int K, int ld, bool transpose, int nt,
                                uint16_t *planes, const int *skip = nullptr);
cudaError_t launch_gemm_planes(const Launch &L, const GemmPlanes &g);
// the single-term planes of a BF16 source
cudaError_t launch_split_planes_bf16(const Launch &L, const void *src, int rows, int K, int ld, bool transpose,
                                     uint16_t *planes, const int *skip = nullptr);
size_t gemm_tc_parts_floats(int M, int N, int ksplit);
cudaError_t launch_sgemm_splitk(const Launch &L, const GemmArgs &g, float *parts, int splits);
size_t sgemm_splitk_parts(int M, int ldc, int splits);
// C = alpha * op(A) op(B) + beta * C in FP64 with float or double operands, split-K slices
// written to C + z * slice_stride (summed by launch_sum_slices).
struct DgemmArgs {
  const void *A;
  const void *B;
  double *C;
  int M, N, K, lda, ldb, ldc;
  bool transA, transB;
  bool a_f32, b_f32;
  double alpha, beta;
  int splits;
  size_t slice_stride;
};
cudaError_t launch_dgemm(const Launch &L, const DgemmArgs &g);
cudaError_t launch_sum_slices(const Launch &L, const double *parts, int splits, size_t slice_stride, size_t n,
                              double *out, double scale);
cudaError_t launch_mirror_lower(const Launch &L, float *A, int n);
cudaError_t launch_f32_to_f64(const Launch &L, const float *x, double *y, size_t n);
cudaError_t launch_f64_to_f32(const Launch &L, const double *x, float *y, size_t n, bool zero_upper, int n_cols);
// Cholesky A = L L^T and L^-1 in FP64 (A is overwritten by L, Linv receives L^-1), n x n;
// the large products of the recursion on the tensor cores (ozaki_tc.cu).
cudaError_t launch_chol_inv(const Launch &L, double *A, double *Linv, int n, double *work);
size_t chol_inv_work_doubles(int n);
// ---- ozaki_tc.cu: FP64-accurate GEMM from exact BF16 slices on the tensor cores ----------
size_t gemm_oz_ws_bytes(int M, int N, int K);
bool gemm_oz_ok(int M, int N, int K);
cudaError_t launch_gemm_oz(const Launch &L, const double *A, int lda, bool transA, const double *B, int ldb,
                           bool transB, double *C, int ldc, int M, int N, int K, double alpha, double beta, void *ws);

// ---- factor.cu --------------------------------------------------------------------------
cudaError_t launch_philox_gaussian(const Launch &L, float *out, size_t n, uint64_t seed);
int trace_partials(int sms);
cudaError_t launch_trace_from_activations(const Launch &L, const void *a, bool bf16, int T, int d, double *part,
                                          double *tr);
cudaError_t launch_small_chol_rinv(const Launch &L, const double *G, int k, double *Rinv);
cudaError_t launch_jacobi(const Launch &L, const double *B, int k, double *evals, double *V);
cudaError_t launch_lowrank_outputs(const Launch &L, const float *Q, int d_in, int k, const double *V,
                                   const double *evals, const double *trace, int rank, float *U, float *mu,
                                   float *sigma);
cudaError_t launch_eye(const Launch &L, float *Q, int n);

}  // namespace gift
