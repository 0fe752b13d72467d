// Rank-r factor refresh in FP32 with its dense products on the tensor cores.
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17): A ~ U_r Lambda_r U_r^T
// with r = 32, refreshed every K = 50 steps (Algorithm 1).  The top eigenpairs come from
// randomised block subspace iteration (N. Halko, P.-G. Martinsson, J. Tropp, "Finding
// structure with randomness", SIAM Review 2011) with k = 64 columns:
//
//   Q = orth(Omega)                       Omega seeded Gaussian (Philox4x32-10)
//   repeat up to q times:
//     Y = A Q                             tensor cores (gemm_tc.cu: exact BF16 splits of A and Q)
//     B = Q^T Y; (theta, V) = eig(B)      Rayleigh-Ritz: 64 x 64, FP32 Jacobi in one CTA
//     stop once the top r Ritz pairs have residuals ||A u - theta u|| <= 1e-4 theta
//     Q = orth(Y V)                       CholQR2 in FP32
//   final Y = A Q, B = Q^T Y, (mu, V) = eig(B), U = Q V[:, :r]
//
// Rotating Y to the Ritz directions before orthonormalising keeps the CholQR input well
// conditioned: A (Q V) is close to (Q V) diag(theta) plus the residuals of the Ritz pairs, so
// its normalised columns are nearly orthogonal and the FP32 Gram matrix (error ~ 2^-24 of the
// column norms) stays safely positive definite.  The start Omega is Gaussian, itself well
// conditioned.  FP32 replaces the FP64 of the small dense steps because this GPU's FP64 rate
// is a small fraction of its FP32 rate.
//
// Every kernel of the loop takes a device flag: once the Ritz values have converged the
// remaining iterations' launches return at once, so the host enqueues a fixed number of
// launches and never waits on the device.
#include <cmath>

#include <cuda_bf16.h>

#include "kernels.cuh"

namespace gift {

namespace {
constexpr int kK = 64;              // sketch columns
constexpr int kGramRows = 32;       // rows staged per step of the tall Gram
}  // namespace

// =====================================================================================
// parts[b] = X[rows of CTA b]^T Y[rows of CTA b] (k x k), X and Y d x k row-major, k <= 64.
// Thread t holds output row t / 4 and 16 columns from 16 (t % 4).  Each sum is compensated
// (the Dot2 scheme of T. Ogita, S. Rump, S. Oishi, "Accurate sum and dot product", SIAM J. Sci.
// Comput. 2005: exact product errors by FMA, exact addition errors by TwoSum), so it is as
// accurate as if it were formed in twice the working precision and then rounded.
// =====================================================================================
__global__ void __launch_bounds__(256) k_gram_tall(const float *__restrict__ X, const float *__restrict__ Y, int d,
                                                   int k, int rows_per_cta, float *__restrict__ parts,
                                                   const int *skip) {
  if (skip && *skip) return;
  __shared__ float sx[kGramRows][kK + 1], sy[kGramRows][kK + 4];
  const int tid = threadIdx.x, i = tid >> 2, j0 = (tid & 3) * 16;
  float acc[16], cmp[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = cmp[q] = 0.0f;
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(d, r0 + rows_per_cta);
  for (int rb = r0; rb < r1; rb += kGramRows) {
    for (int idx = tid; idx < kGramRows * kK; idx += 256) {
      const int rr = idx / kK, c = idx % kK;
      const int row = rb + rr;
      const bool in = row < r1 && c < k;
      sx[rr][c] = in ? X[(size_t)row * k + c] : 0.0f;
      sy[rr][c] = in ? Y[(size_t)row * k + c] : 0.0f;
    }
    __syncthreads();
#pragma unroll 2
    for (int rr = 0; rr < kGramRows; ++rr) {
      const float xv = sx[rr][i];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float yv = sy[rr][j0 + q];
        const float p = __fmul_rn(xv, yv);
        const float pe = fmaf(xv, yv, -p);              // exact error of the product
        const float t = __fadd_rn(acc[q], p);
        const float z = __fsub_rn(t, acc[q]);
        const float e = __fadd_rn(__fsub_rn(acc[q], __fsub_rn(t, z)), __fsub_rn(p, z));   // exact error of the sum
        acc[q] = t;
        cmp[q] = __fadd_rn(cmp[q], __fadd_rn(e, pe));
      }
    }
    __syncthreads();
  }
  if (i < k) {
    float *o = parts + (size_t)blockIdx.x * k * k + (size_t)i * k;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (j0 + q < k) o[j0 + q] = __fadd_rn(acc[q], cmp[q]);
  }
}

// Compensated (TwoSum) accumulation: s + c carries the running sum to twice the precision.
__device__ __forceinline__ void two_sum_add(float &s, float &c, float x) {
  const float t = __fadd_rn(s, x);
  const float z = __fsub_rn(t, s);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(x, z)));
  s = t;
}

// out = the sum of the CTAs' partials (compensated), symmetrised when sym.  Eight threads per
// entry: thread u sums partials u, u + 8, u + 16, ... in order, then thread 0 of the group adds
// the eight sums in thread order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(256) k_gram_sum(const float *__restrict__ parts, int nparts, int k, bool sym,
                                                  float scale, float *__restrict__ out, const int *skip) {
  if (skip && *skip) return;
  const int gid = blockIdx.x * blockDim.x + threadIdx.x;
  const int idx = gid >> 3, sub = gid & 7, lane = threadIdx.x & 31;
  const bool valid = idx < k * k;
  const int i = valid ? idx / k : 0, j = valid ? idx % k : 0;
  const size_t kk = (size_t)k * k;
  float s = 0.0f, c = 0.0f;
  if (valid) {
    for (int p0 = sub; p0 < nparts; p0 += 64) {
      float x[8], y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {   // the loads first, then the dependent sums
        const int p = p0 + 8 * u;
        x[u] = p < nparts ? parts[(size_t)p * kk + idx] : 0.0f;
        y[u] = (sym && p < nparts) ? parts[(size_t)p * kk + (size_t)j * k + i] : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        two_sum_add(s, c, x[u]);
        two_sum_add(s, c, y[u]);
      }
    }
  }
#pragma unroll
  for (int u = 1; u < 8; ++u) {
    const float su = __shfl_sync(0xFFFFFFFFu, s, (lane & ~7) + u);
    const float cu = __shfl_sync(0xFFFFFFFFu, c, (lane & ~7) + u);
    if (sub == 0) {
      two_sum_add(s, c, su);
      c = __fadd_rn(c, cu);
    }
  }
  if (valid && sub == 0) {
    const float v = __fadd_rn(s, c);
    out[idx] = __fmul_rn(sym ? 0.5f * v : v, scale);
  }
}

// =====================================================================================
// Cholesky G = L L^T of a k x k Gram matrix (k = 64), FP32, one CTA of 256 threads; L is
// written lower-triangular (upper part zero).  A pivot below 1e-10 of the largest diagonal (a
// numerically rank-deficient block) is replaced by 1.
// Blocked by panels of 16 columns: warp 0 factors a panel on its own (16 right-looking steps
// on the panel's columns held in registers, two rows per lane, each entry of the pivot column
// passed to the other lanes by a shuffle), then all threads apply the panel's rank-16 update
// to the rows and columns after it; two CTA barriers per panel instead of two per column.
// =====================================================================================
__global__ void __launch_bounds__(256) k_chol32(const float *__restrict__ G, float *__restrict__ Lout,
                                                const int *skip) {
  if (skip && *skip) return;
  __shared__ float S[kK][kK + 1];
  __shared__ float tiny_sh;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int idx = tid; idx < kK * kK; idx += 256) S[idx >> 6][idx & 63] = G[idx];
  if (tid < 32) {   // the largest diagonal entry sets the rank-deficiency floor
    float m = fmaxf(G[tid * kK + tid], G[(tid + 32) * kK + tid + 32]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (tid == 0) tiny_sh = m * 1e-10f + 1e-30f;
  }
  __syncthreads();
  const float tiny = tiny_sh;
  for (int p = 0; p < kK / 16; ++p) {
    const int c0 = 16 * p, c1 = c0 + 16;
    if (tid < 32) {
      // the panel's 16 columns of rows lane and lane + 32 in registers; an entry of column j
      // reaches the other lanes by a shuffle from the lane holding its row
      const int ra = lane, rb = lane + 32;
      float x0[16], x1[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        x0[k] = S[ra][c0 + k];
        x1[k] = S[rb][c0 + k];
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = c0 + jj;
        // 1/sqrt(d) from the hardware estimate and one Newton step, sqrt(d) = d / sqrt(d)
        const float d = __shfl_sync(0xFFFFFFFFu, j < 32 ? x0[jj] : x1[jj], j & 31);
        float rp = 1.0f, piv = 1.0f;
        if (d > tiny) {
          const float q = rsqrtf(d);
          rp = q * fmaf(-0.5f * d * q, q, 1.5f);
          piv = d * rp;
        }
        if (ra > j) x0[jj] *= rp;
        else if (ra == j) x0[jj] = piv;
        if (rb > j) x1[jj] *= rp;
        else if (rb == j) x1[jj] = piv;
        // the panel's columns right of j: S[r][c] -= L[r][j] L[c][j] for r >= c
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          if (cc <= jj) continue;
          const int c = c0 + cc;
          const float lc = __shfl_sync(0xFFFFFFFFu, c < 32 ? x0[jj] : x1[jj], c & 31);
          if (ra >= c) x0[cc] = fmaf(-x0[jj], lc, x0[cc]);
          if (rb >= c) x1[cc] = fmaf(-x1[jj], lc, x1[cc]);
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        S[ra][c0 + k] = x0[k];
        S[rb][c0 + k] = x1[k];
      }
    }
    __syncthreads();
    // trailing update: S[r][c] -= sum over the panel of L[r][k] L[c][k], c1 <= c <= r
    const int m = kK - c1;
    for (int idx = tid; idx < m * m; idx += 256) {
      const int r = c1 + idx / m, c = c1 + idx % m;
      if (c > r) continue;
      float acc = S[r][c];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc = fmaf(-S[r][c0 + k], S[c][c0 + k], acc);
      S[r][c] = acc;
    }
    __syncthreads();
  }
  for (int idx = tid; idx < kK * kK; idx += 256) {
    const int r = idx >> 6, c = idx & 63;
    Lout[idx] = (c <= r) ? S[r][c] : 0.0f;
  }
}

// =====================================================================================
// Symmetric eigensolver, k = 64, FP32, one CTA: one-sided (Hestenes) Jacobi on W = B V.  Each
// round applies 32 disjoint plane rotations to pairs of columns of W and V (a round-robin
// schedule over 64 indices: 63 rounds per sweep, every pair once), warp w taking pair w: the
// warp forms alpha = |W_p|^2, beta = |W_q|^2 and gamma = W_p . W_q with shuffles and rotates
// both columns so that W_p . W_q = 0 (J. Demmel, K. Veselic, "Jacobi's method is more accurate
// than QR", SIAM J. Matrix Anal. Appl. 1992).  One CTA barrier per round.  A pair is rotated
// while |gamma| > 1e-6 sqrt(alpha beta); the solver stops after a sweep that rotates nothing,
// or after max_sweeps (then NOT_CONVERGED, when a status word is given).  At convergence W's
// columns are B's eigenvectors scaled by the eigenvalues: evals[c] = |W_c| with the sign of
// V_c . W_c, descending (ties by index); V's column c is the eigenvector of evals[c].
// =====================================================================================
constexpr int kJ32Threads = 1024;

__global__ void __launch_bounds__(kJ32Threads) k_jacobi32(const float *__restrict__ B, float *__restrict__ evals,
                                                          float *__restrict__ Vout, int max_sweeps, int *status,
                                                          const int *skip) {
  if (skip && *skip) return;
  __shared__ float W[kK][kK + 1], V[kK][kK + 1];
  __shared__ float ev_sh[kK];
  __shared__ int rot[2];   // per sweep parity: whether the sweep rotated anything
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  for (int idx = tid; idx < kK * kK; idx += kJ32Threads) {
    const int i = idx >> 6, j = idx & 63;
    W[i][j] = 0.5f * (B[i * kK + j] + B[j * kK + i]);
    V[i][j] = (i == j) ? 1.0f : 0.0f;
  }
  if (tid < 2) rot[tid] = 0;
  __syncthreads();
  int sweep = 0;
  bool converged = false;
  for (; sweep < max_sweeps; ++sweep) {
    for (int r = 0; r < kK - 1; ++r) {
      const int a = (w == 0) ? kK - 1 : (r + w) % (kK - 1);
      const int b = (w == 0) ? r : (r - w + (kK - 1)) % (kK - 1);
      const int p = min(a, b), q = max(a, b);
      const float wp0 = W[l][p], wp1 = W[l + 32][p], wq0 = W[l][q], wq1 = W[l + 32][q];
      float al = fmaf(wp0, wp0, wp1 * wp1), be = fmaf(wq0, wq0, wq1 * wq1), ga = fmaf(wp0, wq0, wp1 * wq1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        al += __shfl_xor_sync(0xFFFFFFFFu, al, o);
        be += __shfl_xor_sync(0xFFFFFFFFu, be, o);
        ga += __shfl_xor_sync(0xFFFFFFFFu, ga, o);
      }
      // |gamma| > 1e-6 sqrt(alpha beta), squared (no square root on the chain); the same
      // decision in every lane.  The rotation needs no correctly rounded roots or quotients:
      // c and s from the hardware reciprocal square root keep c^2 + s^2 = 1 to a few ulp.
      if (ga * ga > 1e-12f * (al * be) && ga != 0.0f) {
        const float zeta = (be - al) * __frcp_rn(2.0f * ga);
        const float t = copysignf(__frcp_rn(fabsf(zeta) + __fsqrt_rn(fmaf(zeta, zeta, 1.0f))), zeta);
        const float c = rsqrtf(fmaf(t, t, 1.0f)), s = t * c;
        W[l][p] = c * wp0 - s * wq0;
        W[l][q] = s * wp0 + c * wq0;
        W[l + 32][p] = c * wp1 - s * wq1;
        W[l + 32][q] = s * wp1 + c * wq1;
        const float vp0 = V[l][p], vp1 = V[l + 32][p], vq0 = V[l][q], vq1 = V[l + 32][q];
        V[l][p] = c * vp0 - s * vq0;
        V[l][q] = s * vp0 + c * vq0;
        V[l + 32][p] = c * vp1 - s * vq1;
        V[l + 32][q] = s * vp1 + c * vq1;
        if (l == 0) rot[sweep & 1] = 1;
      }
      // the next sweep's flag: every thread read it (as the previous sweep's) before round 0's
      // barrier, and nothing sets it before the next sweep
      if (r == 1 && tid == 0) rot[(sweep + 1) & 1] = 0;
      __syncthreads();
    }
    if (!rot[sweep & 1]) {
      converged = true;
      break;
    }
  }
  if (tid == 0 && !converged && status) set_status(status, GIFT_ERR_NOT_CONVERGED);
  if (w < 2) {   // eigenvalue of column c = tid: |W_c| with the sign of V_c . W_c
    const int c = tid;
    float nn = 0.0f, dv = 0.0f;
    for (int i = 0; i < kK; ++i) {
      nn = fmaf(W[i][c], W[i][c], nn);
      dv = fmaf(V[i][c], W[i][c], dv);
    }
    ev_sh[c] = (dv < 0.0f) ? -sqrtf(nn) : sqrtf(nn);
  }
  __syncthreads();
  if (tid < kK) {   // descending, ties by index
    const int i = tid;
    const float e = ev_sh[i];
    int pos = 0;
    for (int j = 0; j < kK; ++j) {
      const float f = ev_sh[j];
      pos += (f > e) || (f == e && j < i);
    }
    evals[pos] = e;
    for (int row = 0; row < kK; ++row) Vout[row * kK + pos] = V[row][i];
  }
}

// =====================================================================================
// out = X L^-T (X: d x 64 row-major, L: 64 x 64 lower-triangular), i.e. the solution q of
// L q^T = x^T for every row x, by forward substitution: one warp per row, lane l holding
// entries l and l + 32; step c takes q_c from its lane and removes it from the later entries.
// A warp reads its whole row before it writes, so out may be X.
// =====================================================================================
__global__ void __launch_bounds__(256) k_right_trsm64(const float *X, int d, const float *__restrict__ Lm,
                                                      float *out, const int *skip) {
  if (skip && *skip) return;
  __shared__ float Ls[kK][kK + 1];
  __shared__ float rd[kK];
  for (int idx = threadIdx.x; idx < kK * kK; idx += blockDim.x) Ls[idx / kK][idx % kK] = Lm[idx];
  __syncthreads();
  if (threadIdx.x < kK) rd[threadIdx.x] = 1.0f / Ls[threadIdx.x][threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < d; row += warps) {
    float acc0 = X[(size_t)row * kK + lane], acc1 = X[(size_t)row * kK + 32 + lane];
    float q0 = 0.0f, q1 = 0.0f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float qc = __shfl_sync(0xFFFFFFFFu, acc0, c) * rd[c];   // lane c's entry is final
      if (lane == c) q0 = qc;
      if (lane > c) acc0 = fmaf(-qc, Ls[lane][c], acc0);
      acc1 = fmaf(-qc, Ls[32 + lane][c], acc1);
    }
#pragma unroll
    for (int c = 32; c < 64; ++c) {
      const float qc = __shfl_sync(0xFFFFFFFFu, acc1, c - 32) * rd[c];
      if (lane == c - 32) q1 = qc;
      if (lane > c - 32) acc1 = fmaf(-qc, Ls[32 + lane][c], acc1);
    }
    __syncwarp();
    out[(size_t)row * kK + lane] = q0;
    out[(size_t)row * kK + 32 + lane] = q1;
  }
}

// =====================================================================================
// Rotation to the Ritz directions with the Ritz residuals: Y <- Y V in place (Y = A Q, so
// Y V = A (Q V)), and for every column c the partial sum over the CTA's rows of
// ((Y V)[row][c] - theta_c (Q V)[row][c])^2, the squared residual ||A u_c - theta_c u_c||^2 of
// the Ritz pair (theta_c, u_c = (Q V)[:, c]).  One warp per row, lanes c and c + 32.
// =====================================================================================
__global__ void __launch_bounds__(256) k_ritz_rotate(float *Y, const float *__restrict__ Q, int d,
                                                     const float *__restrict__ V, const float *__restrict__ theta,
                                                     float *__restrict__ res_parts, const int *skip) {
  if (skip && *skip) return;
  __shared__ float sv[kK][kK + 1];
  __shared__ float red[8][kK];
  for (int idx = threadIdx.x; idx < kK * kK; idx += blockDim.x) sv[idx / kK][idx % kK] = V[idx];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float t0 = theta[lane], t1 = theta[32 + lane];
  float s0 = 0.0f, s1 = 0.0f;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + warp; row < d; row += warps) {
    const float y0 = Y[(size_t)row * kK + lane], y1 = Y[(size_t)row * kK + 32 + lane];
    const float q0 = Q[(size_t)row * kK + lane], q1 = Q[(size_t)row * kK + 32 + lane];
    float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
#pragma unroll 8
    for (int c = 0; c < 32; ++c) {
      const float yc = __shfl_sync(0xFFFFFFFFu, y0, c), qc = __shfl_sync(0xFFFFFFFFu, q0, c);
      a0 = fmaf(yc, sv[c][lane], a0);
      a1 = fmaf(yc, sv[c][32 + lane], a1);
      b0 = fmaf(qc, sv[c][lane], b0);
      b1 = fmaf(qc, sv[c][32 + lane], b1);
    }
#pragma unroll 8
    for (int c = 0; c < 32; ++c) {
      const float yc = __shfl_sync(0xFFFFFFFFu, y1, c), qc = __shfl_sync(0xFFFFFFFFu, q1, c);
      a0 = fmaf(yc, sv[32 + c][lane], a0);
      a1 = fmaf(yc, sv[32 + c][32 + lane], a1);
      b0 = fmaf(qc, sv[32 + c][lane], b0);
      b1 = fmaf(qc, sv[32 + c][32 + lane], b1);
    }
    __syncwarp();
    Y[(size_t)row * kK + lane] = a0;
    Y[(size_t)row * kK + 32 + lane] = a1;
    const float e0 = fmaf(-t0, b0, a0), e1 = fmaf(-t1, b1, a1);
    s0 = fmaf(e0, e0, s0);
    s1 = fmaf(e1, e1, s1);
  }
  red[warp][lane] = s0;
  red[warp][32 + lane] = s1;
  __syncthreads();
  if (threadIdx.x < kK) {
    float t = 0.0f;
    for (int w = 0; w < 8; ++w) t += red[w][threadIdx.x];
    res_parts[(size_t)blockIdx.x * kK + threadIdx.x] = t;
  }
}

// Convergence: every one of the top r Ritz pairs has ||A u - theta u|| <= 1e-4 theta plus a
// quarter ulp of the largest Ritz value; then *flag = 1 and the remaining iterations' launches
// return at once.  (Below that the FP32 residual is rounding noise: the loop then runs to its
// iteration cap.)
__global__ void __launch_bounds__(1024) k_ritz_check(const float *__restrict__ res_parts, int nparts,
                                                     const float *__restrict__ theta, int r, int *flag) {
  if (*flag) return;
  __shared__ int moved;
  if (threadIdx.x == 0) moved = 0;
  __syncthreads();
  const float top = fabsf(theta[0]);
  const int col = threadIdx.x >> 4, sub = threadIdx.x & 15;   // 16 threads per column
  float s = 0.0f;
  for (int p = sub; p < nparts; p += 16) s += res_parts[(size_t)p * kK + col];
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if (sub == 0 && col < r && !(sqrtf(s) <= 1e-4f * fabsf(theta[col]) + 0.25f * 0x1p-24f * top)) atomicOr(&moved, 1);
  __syncthreads();
  if (threadIdx.x == 0 && !moved) *flag = 1;
}

// tr(A) = (sum of the squares of the activations) / T: compensated FP32 sums per thread and
// per CTA (squares are exact in FP32 for BF16 activations), the CTAs' sums in FP64.
template <typename Src>
__global__ void __launch_bounds__(256) k_sumsq32(const Src *__restrict__ a, size_t n, double *__restrict__ part) {
  __shared__ double red[256];
  constexpr int V = 16 / sizeof(Src);   // elements per 16-byte load
  float s[V], c[V];
#pragma unroll
  for (int u = 0; u < V; ++u) s[u] = c[u] = 0.0f;
  const size_t nv = n / V;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
    const uint4 w = reinterpret_cast<const uint4 *>(a)[i];
    float v[V];
    if constexpr (sizeof(Src) == 2) {
      const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[2 * u] = __uint_as_float(q[u] << 16);
        v[2 * u + 1] = __uint_as_float(q[u] & 0xFFFF0000u);
      }
    } else {
      v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y); v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {   // independent compensated sums, one per lane of the load
      const float p = __fmul_rn(v[u], v[u]);
      two_sum_add(s[u], c[u], p);
      c[u] = __fadd_rn(c[u], fmaf(v[u], v[u], -p));
    }
  }
  double t = 0.0;
#pragma unroll
  for (int u = 0; u < V; ++u) t += (double)s[u] + (double)c[u];
  if (blockIdx.x == 0 && threadIdx.x == 0)   // the tail that does not fill a 16-byte load
    for (size_t i = nv * V; i < n; ++i) {
      float v;
      if constexpr (sizeof(Src) == 2) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a)[i]);
      else v = a[i];
      t += (double)v * (double)v;
    }
  red[threadIdx.x] = t;
  __syncthreads();
  for (int w2 = 128; w2 > 0; w2 >>= 1) {
    if (threadIdx.x < w2) red[threadIdx.x] += red[threadIdx.x + w2];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = red[0];
}

__global__ void k_sum_partials64(const double *__restrict__ part, int nb, double scale, double *out) {
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < nb; ++i) s += part[i];
    out[0] = s * scale;
  }
}

cudaError_t launch_trace_acts32(const Launch &L, const void *a, bool bf16, int T, int d, double *part, int nparts,
                                double *tr) {
  if (!aligned16(a)) return cudaErrorInvalidValue;
  const size_t n = (size_t)T * d;
  if (bf16) k_sumsq32<__nv_bfloat16><<<nparts, 256, 0, L.stream>>>(static_cast<const __nv_bfloat16 *>(a), n, part);
  else k_sumsq32<float><<<nparts, 256, 0, L.stream>>>(static_cast<const float *>(a), n, part);
  k_sum_partials64<<<1, 32, 0, L.stream>>>(part, nparts, 1.0 / (double)T, tr);
  return cudaGetLastError();
}

// tr(A) = sum of the diagonal of the formed A (FP64 sum of FP32 values).
__global__ void k_trace_diag(const float *__restrict__ A, int d, double *tr) {
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < d; i += 256) s += (double)A[(size_t)i * d + i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) tr[0] = red[0];
}

// =====================================================================================
// host side
// =====================================================================================
int refresh_gram_ctas(int sms, int d) {
  int n = (d + 47) / 48;   // at least 48 rows per CTA, at most one CTA per SM
  if (n > sms) n = sms;
  return n < 1 ? 1 : n;
}

cudaError_t launch_gram_tall(const Launch &L, const float *X, const float *Y, int d, int k, float *parts, float *out,
                             bool sym, const int *skip, float scale) {
  const int ctas = refresh_gram_ctas(L.sms, d);
  const int rows = (d + ctas - 1) / ctas;
  k_gram_tall<<<ctas, 256, 0, L.stream>>>(X, Y, d, k, rows, parts, skip);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_gram_sum<<<(8 * k * k + 255) / 256, 256, 0, L.stream>>>(parts, ctas, k, sym, scale, out, skip);
  return cudaGetLastError();
}

cudaError_t launch_chol32(const Launch &L, const float *G, int k, float *Lout, const int *skip) {
  if (k != kK) return cudaErrorInvalidValue;
  k_chol32<<<1, 256, 0, L.stream>>>(G, Lout, skip);
  return cudaGetLastError();
}

cudaError_t launch_jacobi32(const Launch &L, const float *B, int k, float *evals, float *V, int max_sweeps,
                            bool report, const int *skip) {
  if (k != kK) return cudaErrorInvalidValue;
  k_jacobi32<<<1, kJ32Threads, 0, L.stream>>>(B, evals, V, max_sweeps, report ? L.status : nullptr, skip);
  return cudaGetLastError();
}

cudaError_t launch_right_trsm64(const Launch &L, const float *X, int d, const float *Lm, float *out,
                                const int *skip) {
  int grid = (d + 7) / 8;
  if (grid > 4 * L.sms) grid = 4 * L.sms;
  k_right_trsm64<<<grid, 256, 0, L.stream>>>(X, d, Lm, out, skip);
  return cudaGetLastError();
}

int ritz_rotate_ctas(int sms, int d) {
  int g = (d + 7) / 8;
  return g > sms ? sms : (g < 1 ? 1 : g);
}

cudaError_t launch_ritz_rotate(const Launch &L, float *Y, const float *Q, int d, const float *V, const float *theta,
                               float *res_parts, const int *skip) {
  k_ritz_rotate<<<ritz_rotate_ctas(L.sms, d), 256, 0, L.stream>>>(Y, Q, d, V, theta, res_parts, skip);
  return cudaGetLastError();
}

cudaError_t launch_ritz_check(const Launch &L, const float *res_parts, int nparts, const float *theta, int r,
                              int *flag) {
  k_ritz_check<<<1, 1024, 0, L.stream>>>(res_parts, nparts, theta, r, flag);
  return cudaGetLastError();
}

cudaError_t launch_trace_diag(const Launch &L, const float *A, int d, double *tr) {
  k_trace_diag<<<1, 256, 0, L.stream>>>(A, d, tr);
  return cudaGetLastError();
}

}  // namespace gift
