// Rank-r eigen approximation of the K-FAC input factor (libgift factor refresh).
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17): A ~ U_r Lambda_r U_r^T
// keeping the top r eigenpairs (r = 32 in the paper's runs); Algorithm 1 refreshes the
// factor every K = 50 steps.  The eigenpairs come from randomised block subspace iteration
// (N. Halko, P.-G. Martinsson, J. Tropp, "Finding structure with randomness", SIAM Review
// 2011): a seeded Gaussian start, power steps Y = A Q re-orthonormalised by CholQR2
// (Fukaya, Nakatsukasa, Yanagisawa, Yamamoto 2014) with FP64 Gram matrices, and a
// Rayleigh-Ritz step B = Q^T A Q solved by parallel-order cyclic Jacobi in one CTA.
//
// Random numbers: Philox4x32-10 (J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011) with the Box-Muller transform.
#include <cmath>

#include "kernels.cuh"

namespace gift {

static int capped(const Launch &L, size_t work) {
  size_t g = (work + 255) / 256;
  if (g > (size_t)L.sms * 8) g = (size_t)L.sms * 8;
  if (g < 1) g = 1;
  return (int)g;
}

// =====================================================================================
// Philox4x32-10 + Box-Muller
// =====================================================================================
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    U4 n;
    n.x = hi1 ^ c.y ^ k0;
    n.y = lo1;
    n.z = hi0 ^ c.w ^ k1;
    n.w = lo0;
    c = n;
    k0 += W0;
    k1 += W1;
  }
  return c;
}

__device__ __forceinline__ float u01(uint32_t v) {
  // ((v >> 8) + 0.5) * 2^-24 lies strictly inside (0, 1)
  return ((float)(v >> 8) + 0.5f) * 0x1p-24f;
}

__global__ void k_philox_gaussian(float *__restrict__ out, size_t n, uint32_t k0, uint32_t k1) {
  const size_t ncnt = (n + 3) / 4;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t c = (size_t)blockIdx.x * blockDim.x + threadIdx.x; c < ncnt; c += stride) {
    U4 ctr = {(uint32_t)c, (uint32_t)(c >> 32), 0u, 0u};
    const U4 r = philox4x32_10(ctr, k0, k1);
    float s0, c0, s1, c1;
    const float r0 = sqrtf(-2.0f * logf(u01(r.x)));
    const float r1 = sqrtf(-2.0f * logf(u01(r.z)));
    sincospif(2.0f * u01(r.y), &s0, &c0);
    sincospif(2.0f * u01(r.w), &s1, &c1);
    const float z[4] = {r0 * c0, r0 * s0, r1 * c1, r1 * s1};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (4 * c + e < n) out[4 * c + e] = z[e];
  }
}

cudaError_t launch_philox_gaussian(const Launch &L, float *out, size_t n, uint64_t seed) {
  k_philox_gaussian<<<capped(L, (n + 3) / 4), 256, 0, L.stream>>>(out, n, (uint32_t)seed, (uint32_t)(seed >> 32));
  return cudaGetLastError();
}

// =====================================================================================
// tr(A) = (1/T) sum_t sum_i a_ti^2 straight from the activations, in FP64: per-CTA partial
// sums over a fixed grid-stride partition, then one thread adds the partials in order.
// (The trace fixes sigma = (tr A - sum mu) / (d_in - r), a difference of nearly equal
// numbers for steep spectra, so it is not taken from the FP32 diagonal of A.)
// =====================================================================================
template <typename T>
__device__ __forceinline__ double ld64(const T *p, size_t i);
template <>
__device__ __forceinline__ double ld64<float>(const float *p, size_t i) { return (double)p[i]; }
template <>
__device__ __forceinline__ double ld64<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return (double)__bfloat162float(p[i]);
}

template <typename T>
__global__ void __launch_bounds__(256) k_sumsq_partial(const T *__restrict__ a, size_t n, double *__restrict__ part) {
  __shared__ double s[256];
  double acc = 0.0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const double v = ld64<T>(a, i);
    acc = fma(v, v, acc);
  }
  s[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) s[threadIdx.x] += s[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = s[0];
}

__global__ void k_sum_partials(const double *__restrict__ part, int nb, double scale, double *out) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < nb; ++i) s += part[i];
    out[0] = s * scale;
  }
}

int trace_partials(int sms) { return sms * 4; }

cudaError_t launch_trace_from_activations(const Launch &L, const void *a, bool bf16, int T, int d, double *part,
                                          double *tr) {
  const size_t n = (size_t)T * d;
  const int nb = trace_partials(L.sms);
  if (bf16) k_sumsq_partial<__nv_bfloat16><<<nb, 256, 0, L.stream>>>(reinterpret_cast<const __nv_bfloat16 *>(a), n, part);
  else k_sumsq_partial<float><<<nb, 256, 0, L.stream>>>(reinterpret_cast<const float *>(a), n, part);
  k_sum_partials<<<1, 32, 0, L.stream>>>(part, nb, 1.0 / (double)T, tr);
  return cudaGetLastError();
}

__global__ void k_eye(float *Q, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n * n) Q[i] = (i / n == i % n) ? 1.0f : 0.0f;
}

cudaError_t launch_eye(const Launch &L, float *Q, int n) {
  k_eye<<<(n * n + 255) / 256, 256, 0, L.stream>>>(Q, n);
  return cudaGetLastError();
}

// =====================================================================================
// CholQR step: G = R^T R (R upper) -> R^-1, k <= 64, FP64, one CTA.
// A pivot below 1e-30 of the largest diagonal (a rank-deficient sketch) is replaced by 1.
// =====================================================================================
__global__ void __launch_bounds__(256) k_small_chol_rinv(const double *__restrict__ G, int k,
                                                         double *__restrict__ Rinv) {
  extern __shared__ double qr_sm[];   // two 64 x 65 tiles, opt-in size
  double(*S)[65] = reinterpret_cast<double(*)[65]>(qr_sm);
  double(*X)[65] = reinterpret_cast<double(*)[65]>(qr_sm + 64 * 65);
  const int tid = threadIdx.x;
  for (int idx = tid; idx < k * k; idx += 256) S[idx / k][idx % k] = G[idx];
  __syncthreads();
  double scale = 0.0;
  for (int i = 0; i < k; ++i) scale = fmax(scale, S[i][i]);
  const double tiny = scale * 1e-30 + 1e-300;
  __syncthreads();
  for (int j = 0; j < k; ++j) {
    if (tid == 0) {
      const double d = S[j][j];
      S[j][j] = (d > tiny) ? sqrt(d) : 1.0;
    }
    __syncthreads();
    const double piv = S[j][j];
    for (int i = j + 1 + tid; i < k; i += 256) S[i][j] = S[i][j] / piv;
    __syncthreads();
    const int m = k - j - 1;
    for (int idx = tid; idx < m * m; idx += 256) {
      const int i = j + 1 + idx / m, c = j + 1 + idx % m;
      if (c <= i) S[i][c] = fma(-S[i][j], S[c][j], S[i][c]);
    }
    __syncthreads();
  }
  // reciprocals of the pivots once (FP64 division is slow), kept in the unused upper triangle's
  // diagonal-adjacent column k of S (S has 65 columns)
  for (int i = tid; i < k; i += 256) S[i][64] = 1.0 / S[i][i];
  __syncthreads();
  for (int c = tid; c < k; c += 256) {
    for (int i = 0; i < k; ++i) {
      if (i < c) {
        X[i][c] = 0.0;
        continue;
      }
      double s = (i == c) ? 1.0 : 0.0;
      for (int q = c; q < i; ++q) s = fma(-S[i][q], X[q][c], s);
      X[i][c] = s * S[i][64];
    }
  }
  __syncthreads();
  // G = L L^T, R = L^T, so R^-1 = (L^-1)^T
  for (int idx = tid; idx < k * k; idx += 256) {
    const int i = idx / k, j = idx % k;
    Rinv[idx] = X[j][i];
  }
}

cudaError_t launch_small_chol_rinv(const Launch &L, const double *G, int k, double *Rinv) {
  const int smem = 2 * 64 * 65 * (int)sizeof(double);
  cudaError_t e = ensure_dynamic_smem<k_small_chol_rinv>(smem);
  if (e != cudaSuccess) return e;
  k_small_chol_rinv<<<1, 256, smem, L.stream>>>(G, k, Rinv);
  return cudaGetLastError();
}

// =====================================================================================
// Jacobi eigensolver, k <= 64, FP64, one CTA.  Each sweep visits every pair (p, q) once
// in round-robin order: a round applies kk/2 disjoint rotations at once (kk = k rounded up
// to even; a padding index has a zero row and column and never rotates).  A rotation in the
// (p, q) plane with the smaller angle zeroes A[p][q] (Golub & Van Loan, "Matrix
// Computations", sec. 8.5); A <- J^T A J, V <- V J.
// =====================================================================================
constexpr int kJacMax = 64;
constexpr int kJacThreads = 512;
constexpr int kJacSweeps = 60;

__global__ void __launch_bounds__(kJacThreads) k_jacobi(const double *__restrict__ B, int k,
                                                        double *__restrict__ evals, double *__restrict__ Vout,
                                                        int *status) {
  extern __shared__ double sm[];
  double(*A)[kJacMax + 1] = reinterpret_cast<double(*)[kJacMax + 1]>(sm);
  double(*V)[kJacMax + 1] = reinterpret_cast<double(*)[kJacMax + 1]>(sm + kJacMax * (kJacMax + 1));
  __shared__ double cs_c[kJacMax / 2], cs_s[kJacMax / 2];
  __shared__ int pp[kJacMax / 2], qq[kJacMax / 2];
  __shared__ double red_off[kJacThreads], red_tot[kJacThreads];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int kk = k + (k & 1);
  const int np = kk / 2;
  for (int idx = tid; idx < kk * kk; idx += nt) {
    const int i = idx / kk, j = idx % kk;
    double v = 0.0;
    if (i < k && j < k) v = 0.5 * (B[i * k + j] + B[j * k + i]);
    A[i][j] = v;
    V[i][j] = (i == j) ? 1.0 : 0.0;
  }
  __syncthreads();
  int sweep = 0;
  for (; sweep < kJacSweeps; ++sweep) {
    double off = 0.0, tot = 0.0;
    for (int idx = tid; idx < kk * kk; idx += nt) {
      const int i = idx / kk, j = idx % kk;
      const double a2 = A[i][j] * A[i][j];
      tot += a2;
      if (i != j) off += a2;
    }
    red_off[tid] = off;
    red_tot[tid] = tot;
    __syncthreads();
    for (int w = nt / 2; w > 0; w >>= 1) {
      if (tid < w) {
        red_off[tid] += red_off[tid + w];
        red_tot[tid] += red_tot[tid + w];
      }
      __syncthreads();
    }
    const bool converged = red_off[0] <= 1e-30 * red_tot[0];
    __syncthreads();
    if (converged) break;
    for (int r = 0; r < kk - 1; ++r) {
      if (tid < np) {
        int a, b;
        if (tid == 0) {
          a = kk - 1;
          b = r;
        } else {
          a = (r + tid) % (kk - 1);
          b = (r - tid + (kk - 1)) % (kk - 1);
        }
        const int p = min(a, b), q = max(a, b);
        const double apq = A[p][q], app = A[p][p], aqq = A[q][q];
        double c = 1.0, s = 0.0;
        if (apq != 0.0 && fabs(apq) > 1e-18 * sqrt(fabs(app * aqq))) {
          const double theta = (aqq - app) / (2.0 * apq);
          const double t = (theta >= 0.0 ? 1.0 : -1.0) / (fabs(theta) + sqrt(theta * theta + 1.0));
          c = 1.0 / sqrt(t * t + 1.0);
          s = t * c;
        }
        pp[tid] = p;
        qq[tid] = q;
        cs_c[tid] = c;
        cs_s[tid] = s;
      }
      __syncthreads();
      for (int idx = tid; idx < np * kk; idx += nt) {   // rows p and q
        const int pi = idx / kk, j = idx % kk;
        const int p = pp[pi], q = qq[pi];
        const double c = cs_c[pi], s = cs_s[pi];
        const double ap = A[p][j], aq = A[q][j];
        A[p][j] = c * ap - s * aq;
        A[q][j] = s * ap + c * aq;
      }
      __syncthreads();
      for (int idx = tid; idx < np * kk; idx += nt) {   // columns p and q, and V
        const int pi = idx / kk, i = idx % kk;
        const int p = pp[pi], q = qq[pi];
        const double c = cs_c[pi], s = cs_s[pi];
        const double ap = A[i][p], aq = A[i][q];
        A[i][p] = c * ap - s * aq;
        A[i][q] = s * ap + c * aq;
        const double vp = V[i][p], vq = V[i][q];
        V[i][p] = c * vp - s * vq;
        V[i][q] = s * vp + c * vq;
      }
      __syncthreads();
      if (tid < np && cs_s[tid] != 0.0) {
        A[pp[tid]][qq[tid]] = 0.0;
        A[qq[tid]][pp[tid]] = 0.0;
      }
      __syncthreads();
    }
  }
  if (tid == 0 && sweep >= kJacSweeps) set_status(status, GIFT_ERR_NOT_CONVERGED);
  // sort eigenvalues descending (position by comparison count, ties by index)
  for (int i = tid; i < k; i += nt) {
    const double e = A[i][i];
    int pos = 0;
    for (int j = 0; j < k; ++j) {
      const double f = A[j][j];
      pos += (f > e) || (f == e && j < i);
    }
    evals[pos] = e;
    for (int row = 0; row < k; ++row) Vout[row * k + pos] = V[row][i];
  }
}

cudaError_t launch_jacobi(const Launch &L, const double *B, int k, double *evals, double *V) {
  const size_t smem = 2 * sizeof(double) * kJacMax * (kJacMax + 1);
  cudaError_t e = ensure_dynamic_smem<k_jacobi>((int)smem);
  if (e != cudaSuccess) return e;
  k_jacobi<<<1, kJacThreads, smem, L.stream>>>(B, k, evals, V, L.status);
  return cudaGetLastError();
}

// =====================================================================================
// U = Q V[:, :rank] (FP64 dot products), mu = top eigenvalues, sigma = mean of the rest of
// the spectrum: (tr A - sum mu) / (d_in - rank), or 1 when rank == d_in.
// =====================================================================================
__global__ void __launch_bounds__(256) k_lowrank_outputs(const float *__restrict__ Q, int d_in, int k,
                                                         const double *__restrict__ V, const double *__restrict__ ev,
                                                         const double *__restrict__ trace, int rank,
                                                         float *__restrict__ U, float *__restrict__ mu,
                                                         float *__restrict__ sigma, int *status) {
  const size_t n = (size_t)d_in * rank;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += stride) {
    const size_t j = idx / rank;
    const int r = (int)(idx - j * rank);
    double s = 0.0;
    for (int c = 0; c < k; ++c) s = fma((double)Q[j * k + c], V[c * k + r], s);
    U[idx] = (float)s;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    double sum = 0.0;
    bool bad = false;
    for (int r = 0; r < rank; ++r) {
      mu[r] = (float)ev[r];
      sum += ev[r];
      if (!(ev[r] > 0.0) || !((float)ev[r] > 0.0f)) bad = true;
    }
    double sg = 1.0;
    if (rank < d_in) sg = (trace[0] - sum) / (double)(d_in - rank);
    if (!(sg > 0.0) || !((float)sg > 0.0f)) bad = true;
    sigma[0] = (float)sg;
    if (bad) set_status(status, GIFT_ERR_NOT_PD);
  }
}

cudaError_t launch_lowrank_outputs(const Launch &L, const float *Q, int d_in, int k, const double *V,
                                   const double *evals, const double *trace, int rank, float *U, float *mu,
                                   float *sigma) {
  k_lowrank_outputs<<<capped(L, (size_t)d_in * rank), 256, 0, L.stream>>>(Q, d_in, k, V, evals, trace, rank, U,
                                                                          mu, sigma, L.status);
  return cudaGetLastError();
}

}  // namespace gift
