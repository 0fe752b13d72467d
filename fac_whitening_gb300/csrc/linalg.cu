// Dense linear algebra for the factor refresh and the full-rank transforms of libgift.
//
// GIFT reading notes (zhongzhuzhou.org): K-FAC factors A = E[a a^T], G = E[delta delta^T]
// (prerequisites, eq. (4)); Cholesky A = L_A L_A^T, G = L_G L_G^T (core idea step 2, eq. (7));
// whitening W~ = L_G^-1 W L_A^-T (eq. (11)) and map back W^ = L_G X L_A^T (eq. (14)).
//
// k_sgemm   FP32-accumulating GEMM (FP32 or BF16 operands), 128 x {64,128} tiles, split-K,
//           triangular operand skipping and lower-tile-only mode (for a^T a).
// k_dgemm   FP64-accumulating GEMM (FP32 or FP64 operands), split-K.
// chol_inv  recursive blocked Cholesky that also forms L^-1, in FP64:
//             L11 = chol(A11), L21 = A21 L11^-T, S = A22 - L21 L21^T, L22 = chol(S),
//             (L^-1)21 = -L22^-1 L21 L11^-1, with a one-CTA kernel for blocks <= 64.
#include <cmath>

#include "kernels.cuh"

namespace gift {

template <typename T>
__device__ __forceinline__ float ldf(const T *p, size_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}

static int capped_grid(const Launch &L, size_t work) {
  size_t g = (work + 255) / 256;
  if (g > (size_t)L.sms * 8) g = (size_t)L.sms * 8;
  if (g < 1) g = 1;
  return (int)g;
}

// =====================================================================================
// SGEMM: thread (ty, tx) owns rows ty + 16 i (i < 8) and columns 4 tx + 64 n (+0..3).
// =====================================================================================
__device__ __forceinline__ void lower_tile_coords(int lin, int &bm, int &bn) {
  // lin = bm (bm + 1) / 2 + bn with 0 <= bn <= bm
  long long m = (long long)((sqrt(8.0 * (double)lin + 1.0) - 1.0) * 0.5);
  while ((m + 1) * (m + 2) / 2 <= lin) ++m;
  while (m * (m + 1) / 2 > lin) --m;
  bm = (int)m;
  bn = (int)(lin - m * (m + 1) / 2);
}

template <int NC, bool TA, bool TB, typename TAe, typename TBe>
__global__ void __launch_bounds__(256) k_sgemm(GemmArgs g, int kslice, size_t c_slice) {
  constexpr int BM = 128, BN = 64 * NC, BK = 16;
  __shared__ float As[BK][BM + 1];
  __shared__ __align__(16) float Bs[BK][BN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  int m0, n0;
  if (g.lower_tiles) {
    int bm, bn;
    lower_tile_coords(blockIdx.x, bm, bn);
    m0 = bm * BM;
    n0 = bn * BN;
  } else {
    m0 = blockIdx.y * BM;
    n0 = blockIdx.x * BN;
  }
  const TAe *A = reinterpret_cast<const TAe *>(g.A);
  const TBe *B = reinterpret_cast<const TBe *>(g.B);
  const int kbeg = blockIdx.z * kslice;
  int kend = min(g.K, kbeg + kslice);
  if (g.a_lower) kend = min(kend, m0 + BM);
  if (g.b_lower_t) kend = min(kend, n0 + BN);

  float acc[8][NC][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int n = 0; n < NC; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.0f;

  for (int k0 = kbeg; k0 < kend; k0 += BK) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int idx = q * 256 + tid;
      int m, k;
      if (TA) { m = idx & 127; k = idx >> 7; }
      else { k = idx & 15; m = idx >> 4; }
      const int gm = m0 + m, gk = k0 + k;
      float v = 0.0f;
      if (gm < g.M && gk < kend)
        v = TA ? ldf<TAe>(A, (size_t)gk * g.lda + gm) : ldf<TAe>(A, (size_t)gm * g.lda + gk);
      As[k][m] = v;
    }
#pragma unroll
    for (int q = 0; q < NC * 4; ++q) {
      const int idx = q * 256 + tid;
      int n, k;
      if (TB) { k = idx & 15; n = idx >> 4; }
      else { n = idx % BN; k = idx / BN; }
      const int gn = n0 + n, gk = k0 + k;
      float v = 0.0f;
      if (gn < g.N && gk < kend)
        v = TB ? ldf<TBe>(B, (size_t)gn * g.ldb + gk) : ldf<TBe>(B, (size_t)gk * g.ldb + gn);
      Bs[k][n] = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        const float4 b = *reinterpret_cast<const float4 *>(&Bs[k][4 * tx + 64 * n]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i][n][0] = fmaf(a[i], b.x, acc[i][n][0]);
          acc[i][n][1] = fmaf(a[i], b.y, acc[i][n][1]);
          acc[i][n][2] = fmaf(a[i], b.z, acc[i][n][2]);
          acc[i][n][3] = fmaf(a[i], b.w, acc[i][n][3]);
        }
      }
    }
    __syncthreads();
  }
  float *C = g.C + blockIdx.z * c_slice;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= g.M) continue;
#pragma unroll
    for (int n = 0; n < NC; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int gn = n0 + 4 * tx + 64 * n + e;
        if (gn < g.N) C[(size_t)gm * g.ldc + gn] = __fmul_rn(g.alpha, acc[i][n][e]);
      }
  }
}

__global__ void k_sum_slices_f32(const float *__restrict__ parts, int splits, size_t slice, int M, int N, int ld,
                                 float *__restrict__ out) {
  const size_t n = (size_t)M * N;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t r = i / N, c = i - r * N;
    const size_t off = r * ld + c;
    float s = parts[off];
    for (int z = 1; z < splits; ++z) s = __fadd_rn(s, parts[z * slice + off]);
    out[off] = s;
  }
}

template <int NC, bool TA, bool TB>
static void sgemm_types(const Launch &L, dim3 grid, const GemmArgs &g, int kslice, size_t cs) {
  if (g.a_bf16 && g.b_bf16)
    k_sgemm<NC, TA, TB, __nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, L.stream>>>(g, kslice, cs);
  else if (g.a_bf16)
    k_sgemm<NC, TA, TB, __nv_bfloat16, float><<<grid, 256, 0, L.stream>>>(g, kslice, cs);
  else if (g.b_bf16)
    k_sgemm<NC, TA, TB, float, __nv_bfloat16><<<grid, 256, 0, L.stream>>>(g, kslice, cs);
  else
    k_sgemm<NC, TA, TB, float, float><<<grid, 256, 0, L.stream>>>(g, kslice, cs);
}

template <int NC>
static void sgemm_trans(const Launch &L, dim3 grid, const GemmArgs &g, int kslice, size_t cs) {
  if (g.transA) {
    if (g.transB) sgemm_types<NC, true, true>(L, grid, g, kslice, cs);
    else sgemm_types<NC, true, false>(L, grid, g, kslice, cs);
  } else {
    if (g.transB) sgemm_types<NC, false, true>(L, grid, g, kslice, cs);
    else sgemm_types<NC, false, false>(L, grid, g, kslice, cs);
  }
}

static cudaError_t sgemm_grid_launch(const Launch &L, const GemmArgs &g, int NC, int splits, size_t cs, int kslice) {
  const int BM = 128, BN = 64 * NC;
  dim3 grid;
  if (g.lower_tiles) {
    const long long tiles = (long long)((g.M + BM - 1) / BM);
    grid = dim3((unsigned)(tiles * (tiles + 1) / 2), 1, splits);
  } else {
    grid = dim3((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, splits);
  }
  if (NC == 2) sgemm_trans<2>(L, grid, g, kslice, cs);
  else sgemm_trans<1>(L, grid, g, kslice, cs);
  return cudaGetLastError();
}

cudaError_t launch_sgemm(const Launch &L, const GemmArgs &g) {
  const int NC = (g.N <= 64 && !g.lower_tiles) ? 1 : 2;
  return sgemm_grid_launch(L, g, NC, 1, 0, g.K);
}

size_t sgemm_splitk_parts(int M, int ldc, int splits) { return (size_t)splits * M * ldc; }

// Split-K SGEMM: partial products into `parts` (splits slices of M x ldc), then summed in
// slice order into g.C.  Used for tall-skinny products with few output tiles.
cudaError_t launch_sgemm_splitk(const Launch &L, const GemmArgs &g, float *parts, int splits) {
  const int NC = (g.N <= 64) ? 1 : 2;
  int kslice = (g.K + splits - 1) / splits;
  kslice = (kslice + 15) / 16 * 16;
  const int used = (g.K + kslice - 1) / kslice;
  GemmArgs gp = g;
  gp.C = parts;
  const size_t cs = (size_t)g.M * g.ldc;
  cudaError_t e = sgemm_grid_launch(L, gp, NC, used, cs, kslice);
  if (e != cudaSuccess) return e;
  k_sum_slices_f32<<<capped_grid(L, (size_t)g.M * g.N), 256, 0, L.stream>>>(parts, used, cs, g.M, g.N, g.ldc, g.C);
  return cudaGetLastError();
}

// =====================================================================================
// DGEMM (FP64 accumulate): 64 x 64 tiles, 256 threads, 4 x 4 per thread.
// =====================================================================================
template <typename T>
__device__ __forceinline__ double ldd(const T *p, size_t i) { return (double)p[i]; }

template <bool TA, bool TB, typename TAe, typename TBe>
__global__ void __launch_bounds__(256) k_dgemm(DgemmArgs g, int kslice) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ double As[BK][BM + 1];
  __shared__ double Bs[BK][BN + 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const TAe *A = reinterpret_cast<const TAe *>(g.A);
  const TBe *B = reinterpret_cast<const TBe *>(g.B);
  const int kbeg = blockIdx.z * kslice;
  const int kend = min(g.K, kbeg + kslice);
  double acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0;
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = q * 256 + tid;
      int m, k;
      if (TA) { m = idx & 63; k = idx >> 6; }
      else { k = idx & 15; m = idx >> 4; }
      const int gm = m0 + m, gk = k0 + k;
      double v = 0.0;
      if (gm < g.M && gk < kend) v = TA ? ldd<TAe>(A, (size_t)gk * g.lda + gm) : ldd<TAe>(A, (size_t)gm * g.lda + gk);
      As[k][m] = v;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = q * 256 + tid;
      int n, k;
      if (TB) { k = idx & 15; n = idx >> 4; }
      else { n = idx & 63; k = idx >> 6; }
      const int gn = n0 + n, gk = k0 + k;
      double v = 0.0;
      if (gn < g.N && gk < kend) v = TB ? ldd<TBe>(B, (size_t)gn * g.ldb + gk) : ldd<TBe>(B, (size_t)gk * g.ldb + gn);
      Bs[k][n] = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      double a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  double *C = g.C + blockIdx.z * g.slice_stride;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn >= g.N) continue;
      const size_t o = (size_t)gm * g.ldc + gn;
      const double v = g.alpha * acc[i][j];
      C[o] = (g.beta == 0.0) ? v : fma(g.beta, C[o], v);
    }
  }
}

template <bool TA, bool TB>
static void dgemm_types(const Launch &L, dim3 grid, const DgemmArgs &g, int kslice) {
  if (g.a_f32 && g.b_f32) k_dgemm<TA, TB, float, float><<<grid, 256, 0, L.stream>>>(g, kslice);
  else if (g.a_f32) k_dgemm<TA, TB, float, double><<<grid, 256, 0, L.stream>>>(g, kslice);
  else if (g.b_f32) k_dgemm<TA, TB, double, float><<<grid, 256, 0, L.stream>>>(g, kslice);
  else k_dgemm<TA, TB, double, double><<<grid, 256, 0, L.stream>>>(g, kslice);
}

cudaError_t launch_dgemm(const Launch &L, const DgemmArgs &g) {
  const int splits = g.splits < 1 ? 1 : g.splits;
  const int kslice = (g.K + splits - 1) / splits;
  dim3 grid((g.N + 63) / 64, (g.M + 63) / 64, splits);
  if (g.transA) {
    if (g.transB) dgemm_types<true, true>(L, grid, g, kslice);
    else dgemm_types<true, false>(L, grid, g, kslice);
  } else {
    if (g.transB) dgemm_types<false, true>(L, grid, g, kslice);
    else dgemm_types<false, false>(L, grid, g, kslice);
  }
  return cudaGetLastError();
}

__global__ void k_sum_slices(const double *__restrict__ parts, int splits, size_t slice, size_t n,
                             double *__restrict__ out, double scale) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    double s = 0.0;
    for (int z = 0; z < splits; ++z) s += parts[z * slice + i];
    out[i] = s * scale;
  }
}

cudaError_t launch_sum_slices(const Launch &L, const double *parts, int splits, size_t slice_stride, size_t n,
                              double *out, double scale) {
  k_sum_slices<<<capped_grid(L, n), 256, 0, L.stream>>>(parts, splits, slice_stride, n, out, scale);
  return cudaGetLastError();
}

// =====================================================================================
// small element-wise kernels
// =====================================================================================
__global__ void k_mirror_lower(float *A, int n) {
  __shared__ float t[32][33];
  const int bi = blockIdx.y, bj = blockIdx.x;
  if (bj > bi) return;
  const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int i = bi * 32 + r, j = bj * 32 + tx;
    t[r][tx] = (i < n && j < n) ? A[(size_t)i * n + j] : 0.0f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    // the transpose of lower tile (bi, bj) goes to upper tile (bj, bi)
    const int i = bj * 32 + r, j = bi * 32 + tx;
    if (i < n && j < n && j > i) A[(size_t)i * n + j] = t[tx][r];
  }
}

cudaError_t launch_mirror_lower(const Launch &L, float *A, int n) {
  dim3 grid((n + 31) / 32, (n + 31) / 32), block(32, 8);
  k_mirror_lower<<<grid, block, 0, L.stream>>>(A, n);
  return cudaGetLastError();
}

__global__ void k_f32_to_f64(const float *__restrict__ x, double *__restrict__ y, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) y[i] = (double)x[i];
}
__global__ void k_f64_to_f32(const double *__restrict__ x, float *__restrict__ y, size_t n, bool zero_upper,
                             int ncols) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = (float)x[i];
    if (zero_upper) {
      const size_t r = i / ncols, c = i - r * ncols;
      if (c > r) v = 0.0f;
    }
    y[i] = v;
  }
}

cudaError_t launch_f32_to_f64(const Launch &L, const float *x, double *y, size_t n) {
  k_f32_to_f64<<<capped_grid(L, n), 256, 0, L.stream>>>(x, y, n);
  return cudaGetLastError();
}
cudaError_t launch_f64_to_f32(const Launch &L, const double *x, float *y, size_t n, bool zero_upper, int n_cols) {
  k_f64_to_f32<<<capped_grid(L, n), 256, 0, L.stream>>>(x, y, n, zero_upper, n_cols);
  return cudaGetLastError();
}

// =====================================================================================
// Cholesky + inverse, FP64
// =====================================================================================
constexpr int kCholBase = 64;

// One CTA: factor the n x n (n <= 64) block at A (leading dimension lda) in place into L
// (upper part zeroed) and write L^-1 (lower, upper zeroed) at Li (leading dimension ldl).
// Right-looking: step j takes the pivot, scales column j of L and row j of X (X = I becomes
// L^-1 by forward elimination alongside), then updates every row below j: S_ic for
// j < c <= i and X_ic for c <= j, spread over all threads.  One
// reciprocal square root per step; the rest are multiplications and fused multiply-adds.
__global__ void __launch_bounds__(256) k_chol_inv_small(double *A, int lda, double *Li, int ldl, int n, int *status) {
  extern __shared__ double chol_sm[];   // two (kCholBase x kCholBase+1) tiles, opt-in size
  double(*S)[kCholBase + 1] = reinterpret_cast<double(*)[kCholBase + 1]>(chol_sm);
  double(*X)[kCholBase + 1] = reinterpret_cast<double(*)[kCholBase + 1]>(chol_sm + kCholBase * (kCholBase + 1));
  __shared__ int bad;
  __shared__ double rp_sh;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  for (int idx = tid; idx < n * n; idx += 256) {
    const int i = idx / n, j = idx - i * n;
    S[i][j] = A[(size_t)i * lda + j];
    X[i][j] = (i == j) ? 1.0 : 0.0;
  }
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    if (tid == 0) {
      // 1/sqrt(d) from the FP32 estimate and two Newton steps in FP64 (24 -> 48 -> 96 bits),
      // cheaper on this GPU than its FP64 square root and division
      const double d = S[j][j];
      double piv = 1.0, r = 1.0;
      if (!(d > 0.0)) {
        bad = 1;
      } else {
        r = (double)rsqrtf((float)d);
        if (!(r > 0.0) || isinf(r)) r = 1.0 / sqrt(d);   // d beyond FP32 range
        const double hd = 0.5 * d;
        r = r * fma(-hd, r * r, 1.5);
        r = r * fma(-hd, r * r, 1.5);
        piv = d * r;
      }
      S[j][j] = piv;
      rp_sh = r;
    }
    __syncthreads();
    const double rp = rp_sh;
    if (tid > j && tid < n) S[tid][j] *= rp;            // column j of L
    if (tid < 64 && tid <= j) X[j][tid] *= rp;         // row j of L^-1
    __syncthreads();
    // thread t: column t % 64 of rows j + 1 + t / 64, then every fourth row, from the first
    // row that has the column (c <= i)
    const int c = tid & 63;
    if (c < n) {
      const bool upd_s = c > j;
      const double pivc = upd_s ? S[c][j] : X[j][c];
      int i = j + 1 + (tid >> 6);
      if (i < c) i += ((c - i + 3) >> 2) << 2;
      for (; i < n; i += 4) {
        const double lij = S[i][j];
        if (upd_s) S[i][c] = fma(-lij, pivc, S[i][c]);
        else X[i][c] = fma(-lij, pivc, X[i][c]);
      }
    }
    __syncthreads();
  }
  for (int idx = tid; idx < n * n; idx += 256) {
    const int i = idx / n, j = idx - i * n;
    A[(size_t)i * lda + j] = (j <= i) ? S[i][j] : 0.0;
    Li[(size_t)i * ldl + j] = (j <= i) ? X[i][j] : 0.0;
  }
  if (tid == 0 && bad) set_status(status, GIFT_ERR_NOT_PD);
}

// dst = scale * src on a rows x cols block; scale == 0 writes zeros without reading src.
__global__ void k_copy_block(const double *src, int lds, double *dst, int ldd, int rows, int cols, double scale) {
  const size_t n = (size_t)rows * cols;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t r = i / cols, c = i - r * cols;
    dst[r * ldd + c] = (scale == 0.0) ? 0.0 : (scale == 1.0) ? src[r * lds + c] : scale * src[r * lds + c];
  }
}

static cudaError_t copy_block(const Launch &L, const double *src, int lds, double *dst, int ldd, int rows, int cols,
                              double scale) {
  k_copy_block<<<capped_grid(L, (size_t)rows * cols), 256, 0, L.stream>>>(src, lds, dst, ldd, rows, cols, scale);
  return cudaGetLastError();
}

static cudaError_t dgemm_dd(const Launch &L, const double *A, int lda, bool tA, const double *B, int ldb, bool tB,
                            double *C, int ldc, int M, int N, int K, double alpha, double beta) {
  DgemmArgs g{};
  g.A = A; g.B = B; g.C = C;
  g.M = M; g.N = N; g.K = K; g.lda = lda; g.ldb = ldb; g.ldc = ldc;
  g.transA = tA; g.transB = tB; g.a_f32 = false; g.b_f32 = false;
  g.alpha = alpha; g.beta = beta; g.splits = 1; g.slice_stride = 0;
  return launch_dgemm(L, g);
}

// The recursion's products: on the tensor cores with FP64 accuracy (exact BF16 slices) when a
// workspace is given and the product is large, else the FP64 SIMT GEMM.
static cudaError_t gemm_f64(const Launch &L, const double *A, int lda, bool tA, const double *B, int ldb, bool tB,
                            double *C, int ldc, int M, int N, int K, double alpha, double beta, void *oz) {
  if (oz && M >= 64 && N >= 64 && K >= 64 && gemm_oz_ok(M, N, K))
    return launch_gemm_oz(L, A, lda, tA, B, ldb, tB, C, ldc, M, N, K, alpha, beta, oz);
  return dgemm_dd(L, A, lda, tA, B, ldb, tB, C, ldc, M, N, K, alpha, beta);
}

// Recursive step on the n x n diagonal block at offset `o` of the full matrices (leading
// dimension ld).
static cudaError_t chol_inv_rec(const Launch &L, double *A, double *Li, int ld, int o, int n, double *work,
                                void *oz) {
  double *Ab = A + (size_t)o * ld + o;
  double *Lb = Li + (size_t)o * ld + o;
  if (n <= kCholBase) {
    const int smem = 2 * kCholBase * (kCholBase + 1) * (int)sizeof(double);
    cudaError_t e0 = ensure_dynamic_smem<k_chol_inv_small>(smem);
    if (e0 != cudaSuccess) return e0;
    k_chol_inv_small<<<1, 256, smem, L.stream>>>(Ab, ld, Lb, ld, n, L.status);
    return cudaGetLastError();
  }
  int n1 = ((n / 2 + kCholBase - 1) / kCholBase) * kCholBase;
  if (n1 >= n) n1 = n - kCholBase;
  const int n2 = n - n1;
  cudaError_t e;
  if ((e = chol_inv_rec(L, A, Li, ld, o, n1, work, oz)) != cudaSuccess) return e;
  double *A21 = Ab + (size_t)n1 * ld;          // n2 x n1
  double *A22 = A21 + n1;                      // n2 x n2
  double *L11i = Lb;                           // n1 x n1
  // L21 = A21 L11^-T  (into work, then back into A21)
  if ((e = gemm_f64(L, A21, ld, false, L11i, ld, true, work, n1, n2, n1, n1, 1.0, 0.0, oz)) != cudaSuccess) return e;
  if ((e = copy_block(L, work, n1, A21, ld, n2, n1, 1.0)) != cudaSuccess) return e;
  // S = A22 - L21 L21^T
  if ((e = gemm_f64(L, A21, ld, false, A21, ld, true, A22, ld, n2, n2, n1, -1.0, 1.0, oz)) != cudaSuccess) return e;
  if ((e = chol_inv_rec(L, A, Li, ld, o + n1, n2, work, oz)) != cudaSuccess) return e;
  // (L^-1)21 = -L22^-1 (L21 L11^-1)
  double *L22i = Lb + (size_t)n1 * ld + n1;
  double *Li21 = Lb + (size_t)n1 * ld;
  if ((e = gemm_f64(L, A21, ld, false, L11i, ld, false, work, n1, n2, n1, n1, 1.0, 0.0, oz)) != cudaSuccess) return e;
  if ((e = gemm_f64(L, L22i, ld, false, work, n1, false, Li21, ld, n2, n1, n2, -1.0, 0.0, oz)) != cudaSuccess)
    return e;
  // upper blocks are zero
  if ((e = copy_block(L, nullptr, 0, Ab + n1, ld, n1, n2, 0.0)) != cudaSuccess) return e;
  return copy_block(L, nullptr, 0, Lb + n1, ld, n1, n2, 0.0);
}

// The FP64 scratch of the recursion, then (256-byte aligned) the tensor-core products' slices:
// every product of the recursion has M, N, K <= n / 2 + 64.
static size_t chol_base_doubles(int n) { return (size_t)n * n / 2 + (size_t)kCholBase * n + 64; }
static size_t chol_oz_doubles(int n) {
  if (n <= kCholBase) return 0;
  const int h = n / 2 + 128;
  return gemm_oz_ws_bytes(h, h, h) / 8 + 64;
}

size_t chol_inv_work_doubles(int n) { return chol_base_doubles(n) + chol_oz_doubles(n); }

cudaError_t launch_chol_inv(const Launch &L, double *A, double *Linv, int n, double *work) {
  void *oz = nullptr;
  if (chol_oz_doubles(n) > 0) {
    uintptr_t p = reinterpret_cast<uintptr_t>(work + chol_base_doubles(n));
    oz = reinterpret_cast<void *>((p + 255) & ~(uintptr_t)255);
  }
  return chol_inv_rec(L, A, Linv, n, 0, n, work, oz);
}

}  // namespace gift
