// FP64-accurate matrix products on the 5th-generation tensor cores, for the Cholesky factors
// of the K-FAC matrices (GIFT reading notes, core idea step 2, eq. (7): A = L_A L_A^T, and its
// inverse; refreshed every K steps by Algorithm 1).  This GPU's FP64 units are a small fraction
// of its tensor throughput, and the factor must stay FP64-accurate: the 300M-like layer's A has
// a condition number of about 3e6, so an FP32-accurate factor would be far from the FP64 one.
//
// Splitting.  Following the error-free splitting of K. Ozaki, T. Ogita, S. Oishi and S. M. Rump
// ("Error-free transformations of matrix multiplication by using fast routines of matrix
// multiplication and its applications", Numerical Algorithms 59, 2012), every row r of op(A)
// (M x K) and of op(B)^T (N x K) is scaled by 2^-e_r, e_r the smallest exponent with
// max_k |x_rk| < 2^e_r, and written as seven signed digits of 8 bits:
//
//   x_rk 2^-e_r = sum_{s=0..6} d_s 2^{-8(s+1)} + rest,   |rest| <= 2^-57.
//
// The digits come from the integer N = round(|x| 2^(56 - e_r)) < 2^56, built from the FP64
// bit pattern with integer shifts (this GPU's FP64 units are slow), taken 8 bits at a time
// from the least significant end with balanced digits (a digit of 128 or more becomes
// digit - 256 with a carry), and given x's sign: d_0 in [-256, 256], d_s in [-128, 127] for
// s >= 1.  Each digit is an integer of at most 8 significant bits, so it is exact in BF16, and
// the product of two digits is exact in the tensor core.
//
// Levels.  The products d_s(a) d_t(b) with s + t = l share the weight 2^{-8(l + 2)}; the 28
// products with l <= 6 are kept (the rest weigh below 2^-64 of |a|max |b|max).  Over one
// 64-wide K chunk a level's sum is an integer of magnitude at most 2.25 * 2^22 < 2^24, exactly
// representable in FP32, so the tensor core's FP32 accumulation of it is exact whatever its
// internal order.  The epilogue converts each level's chunk sum to an integer and adds it to
// 32-bit integer accumulators (exact for K <= 8192), and only at the end of the tile combines
// the seven levels (as two exact 64-bit fixed-point integers, converted to FP64 and added with
// one FMA) and applies the row and column scales (exact powers of two): the result is the
// product of the sliced operands up to a few FP64 roundings, and the slicing itself keeps 56
// bits of every operand relative to its row maximum.
//
//   k_oz_rowmax   max |x| of every row of op(A) or op(B)^T (bit patterns, atomicMax)
//   k_oz_slices   the seven digit planes (BF16, the blocked layout of gemm_tc.cu: every
//                 128-row x 64-K tile 16 KB of consecutive memory)
//   k_gemm_oz     persistent over 128 x 32 tiles of C.  Warp 8 streams, for each K chunk
//                 and each A digit s, the A digit tile and B's digits 0 .. 6 - s (stacked,
//                 32 rows each) through a 4-stage TMA ring; warp 9 issues one MMA per K step
//                 of 16 with N = 32 (7 - s) into the accumulator columns of levels s .. 6
//                 (the stacked B's row block t lands at level s + t); warps 0-7 add each
//                 chunk's seven level sums into integer registers and write
//                 C = alpha (A B) + beta C in FP64 after the tile's last chunk.
// Every mbarrier wait is clock-bounded and reports GIFT_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

bool plane_map(CUtensorMap *m, const uint16_t *base, uint64_t rows_total, uint32_t box_rows);

namespace {

constexpr int kOzS = 7;                       // digits per operand, levels 0 .. 6
constexpr int kOzM = 128, kOzN = 32, kOzK = 64;
constexpr int kOzATile = kOzM * 128;          // bytes: 128 rows x 64 BF16
constexpr int kOzBTile = kOzN * 128;          // 32 rows x 64 BF16
constexpr int kOzStageBytes = kOzATile + kOzS * kOzBTile;   // 44 KB (a multiple of 1 KB)
constexpr int kOzStages = 4;
constexpr int kOzEpiWarps = 8;
constexpr int kOzThreads = 32 * (kOzEpiWarps + 2);
constexpr uint32_t kOzAccCols = 256;          // TMEM columns per accumulator set (7 x 32 used)
constexpr long long kOzWait = 4000000000LL;   // about two seconds of SM clock
constexpr int kOzMaxK = 8192;                 // integer accumulators exact up to here

struct OzParams {
  int M, N, K;
  int tiles_m, tiles_n, nch;
  int tiles_ra, tiles_rb;   // 128-row tiles of one digit plane of A and of B
  double alpha, beta;
  double *C;
  int ldc;
  const unsigned long long *rmA, *rmB;   // row maxima (bit patterns of |x|)
};

// The row's scale exponent: the smallest e with max |x| < 2^e (0 for an all-zero row), from
// the bit pattern of the maximum (integer arithmetic; subnormal maxima take the library path).
__device__ __forceinline__ int oz_exp(unsigned long long bits) {
  const int ex = (int)((bits >> 52) & 0x7FF);
  if (ex) return ex - 1022;   // 2^(ex-1023) <= m < 2^(ex-1022)
  const double m = __longlong_as_double((long long)bits);
  return (m == 0.0) ? 0 : ilogb(m) + 1;
}

// 2^e as a double (exact), from the exponent bits where e is a normal exponent.
__device__ __forceinline__ double oz_pow2(int e) {
  if (e >= -1022 && e <= 1023) return __longlong_as_double((long long)(e + 1023) << 52);
  return ldexp(1.0, e);
}

template <bool TRANS>
__device__ __forceinline__ double oz_ld(const double *src, int rows, int K, int ld, int r, int k) {
  if (r >= rows || k >= K) return 0.0;
  return TRANS ? src[(size_t)k * ld + r] : src[(size_t)r * ld + k];
}

}  // namespace

// 32 rows x 64 K per block of 256 threads, staged through shared memory (coalesced along K,
// or along the rows when the source is transposed).
template <bool TRANS>
__global__ void __launch_bounds__(256) k_oz_rowmax(const double *__restrict__ src, int rows, int K, int ld,
                                                   unsigned long long *__restrict__ rmax) {
  __shared__ unsigned long long tile[32][64 + 1];
  const int r0 = blockIdx.y * 32, k0 = blockIdx.x * 64, tid = threadIdx.x;
  for (int q = tid; q < 32 * 64; q += 256) {
    int r, k;
    if (TRANS) {
      k = q >> 5;
      r = q & 31;
    } else {
      r = q >> 6;
      k = q & 63;
    }
    // |x| as its bit pattern: for non-negative doubles the integer order is the value order
    tile[r][k] = (unsigned long long)__double_as_longlong(oz_ld<TRANS>(src, rows, K, ld, r0 + r, k0 + k)) &
                 0x7FFFFFFFFFFFFFFFull;
  }
  __syncthreads();
  const int r = tid >> 3, kb = (tid & 7) * 8;
  unsigned long long m = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) m = max(m, tile[r][kb + u]);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) m = max(m, (unsigned long long)__shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((tid & 7) == 0 && r0 + r < rows && m > 0) atomicMax(rmax + r0 + r, m);
}

// The seven digit planes; thread = one row, 8 consecutive K.
template <bool TRANS>
__global__ void __launch_bounds__(256) k_oz_slices(const double *__restrict__ src, int rows, int K, int ld,
                                                   int rows_pad, int ldk, const unsigned long long *__restrict__ rmax,
                                                   uint16_t *__restrict__ planes) {
  __shared__ double tile[32][64 + 1];
  const int r0 = blockIdx.y * 32, k0 = blockIdx.x * 64, tid = threadIdx.x;
  for (int q = tid; q < 32 * 64; q += 256) {
    int r, k;
    if (TRANS) {
      k = q >> 5;
      r = q & 31;
    } else {
      r = q >> 6;
      k = q & 63;
    }
    tile[r][k] = oz_ld<TRANS>(src, rows, K, ld, r0 + r, k0 + k);
  }
  __syncthreads();
  const int r = tid >> 3, kb = (tid & 7) * 8;
  const int gr = r0 + r;
  const int e = (gr < rows) ? oz_exp(rmax[gr]) : 0;
  uint32_t w[kOzS][4];
#pragma unroll
  for (int u = 0; u < 8; u += 2) {
    float d[2][kOzS];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const unsigned long long bits = (unsigned long long)__double_as_longlong(tile[r][kb + u + h]);
      const int ex = (int)((bits >> 52) & 0x7FF);
      // |x| = sig 2^(ex - 1075) (subnormals: ex = 0, exponent -1074); N = round(|x| 2^(56 - e))
      const unsigned long long sig = (bits & 0xFFFFFFFFFFFFFull) | (ex ? (1ull << 52) : 0ull);
      const int sh = (ex ? ex : 1) - 1075 + 56 - e;   // N = sig 2^sh, sh <= 4 since |x| < 2^e
      unsigned long long nn;
      if (sh >= 0) nn = sig << sh;
      else if (sh > -64) nn = (sig + (1ull << (-sh - 1))) >> (-sh);   // round half up
      else nn = 0;
      const float sgn = (bits >> 63) ? -1.0f : 1.0f;
#pragma unroll
      for (int q = kOzS - 1; q >= 1; --q) {   // balanced base-256 digits, least significant first
        int dg = (int)(nn & 255u);
        nn >>= 8;
        if (dg >= 128) {
          dg -= 256;
          nn += 1;
        }
        d[h][q] = sgn * (float)dg;
      }
      d[h][0] = sgn * (float)nn;   // 0 .. 256
    }
#pragma unroll
    for (int s = 0; s < kOzS; ++s) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(d[0][s]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(d[1][s]));
      w[s][u >> 1] = lo | (hi << 16);
    }
  }
  const size_t off = ((size_t)(gr >> 7) * (ldk >> 6) + (k0 >> 6)) * 8192 + (size_t)(gr & 127) * 64 + kb;
  const size_t plane = (size_t)rows_pad * ldk;
#pragma unroll
  for (int s = 0; s < kOzS; ++s)
    *reinterpret_cast<uint4 *>(planes + (size_t)s * plane + off) = make_uint4(w[s][0], w[s][1], w[s][2], w[s][3]);
}

__global__ void __launch_bounds__(kOzThreads, 1) k_gemm_oz(const __grid_constant__ OzParams P,
                                                           const __grid_constant__ CUtensorMap tmA,
                                                           const __grid_constant__ CUtensorMap tmB, int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[kOzStages], empty[kOzStages], afull[2], aempty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 2 * kOzAccCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kOzStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&afull[a], 1);
      tc::mbar_init(&aempty[a], kOzEpiWarps);
    }
    tc::fence_mbar_init();
    failed = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const int ntiles = P.tiles_m * P.tiles_n;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (failed) return false;
    if (!tc::mbar_wait_bounded(bar, parity, kOzWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kOzEpiWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tensormap(&tmA);
      tc::prefetch_tensormap(&tmB);
      int s = 0, phase = 0;
      long long g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const int tm = t / P.tiles_n, tn = t - tm * P.tiles_n;
        const int tb = (tn * kOzN) >> 7, sub = (tn * kOzN) & 127;
        for (int c = 0; c < P.nch && ok; ++c) {
          for (int da = 0; da < kOzS; ++da) {
            if (!(ok = wait(&empty[s], (uint32_t)(phase ^ 1)))) break;
            uint8_t *st = sm + (size_t)s * kOzStageBytes;
            tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(kOzATile + (kOzS - da) * kOzBTile));
            tc::tma_load_2d(st, &tmA, 0, ((da * P.tiles_ra + tm) * P.nch + c) * 128, &full[s]);
            for (int db = 0; db < kOzS - da; ++db)
              tc::tma_load_2d(st + kOzATile + db * kOzBTile, &tmB, 0, ((db * P.tiles_rb + tb) * P.nch + c) * 128 + sub,
                              &full[s]);
            ++g;
            if (++s == kOzStages) {
              s = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (failed) {   // let this CTA's loads land before the shared memory is released
        for (int q = 0; q < kOzStages; ++q) {
          const long long n = g / kOzStages + (q < (int)(g % kOzStages) ? 1 : 0);
          if (n) tc::mbar_wait_bounded(&full[q], (uint32_t)((n - 1) & 1), kOzWait);
        }
      }
    }
  } else if (warp == kOzEpiWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int s = 0, phase = 0, a = 0, aphase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        for (int c = 0; c < P.nch && ok; ++c) {
          if (!(ok = wait(&aempty[a], (uint32_t)(aphase ^ 1)))) break;
          for (int da = 0; da < kOzS; ++da) {
            if (!(ok = wait(&full[s], (uint32_t)phase))) break;
            tc::fence_after_sync();
            const uint32_t base = tc::smem_u32(sm + (size_t)s * kOzStageBytes);
            const uint32_t bb = base + kOzATile;
            const uint32_t d = tmem + (uint32_t)(a * kOzAccCols + kOzN * da);
            const uint32_t idesc = tc::idesc_bf16(kOzM, kOzN * (kOzS - da));
#pragma unroll
            for (int k = 0; k < kOzK / 16; ++k)
              tc::mma_bf16(d, tc::sdesc_kmajor_sw128(base + 32 * k), tc::sdesc_kmajor_sw128(bb + 32 * k), idesc,
                           (da > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(&empty[s]);
            if (++s == kOzStages) {
              s = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          tc::mma_commit(&afull[a]);
          a ^= 1;
          if (a == 0) aphase ^= 1;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 0-7): 32 rows x 16 columns of every level ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int a = 0, aphase = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const int tm = t / P.tiles_n, tn = t - tm * P.tiles_n;
      int acc[kOzS][16];
#pragma unroll
      for (int l = 0; l < kOzS; ++l)
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[l][j] = 0;
      bool ok = true;
      for (int c = 0; c < P.nch; ++c) {
        if (!(ok = wait(&afull[a], (uint32_t)aphase))) break;
        tc::fence_after_sync();
        const uint32_t col = tmem + lane_off + (uint32_t)(a * kOzAccCols + 16 * half);
#pragma unroll
        for (int l = 0; l < kOzS; ++l) {
          uint32_t r0[16];
          tc::tmem_ld16_nowait(col + kOzN * l, r0);
          tc::tmem_wait_ld16(r0);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[l][j] += __float2int_rz(__uint_as_float(r0[j]));
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&aempty[a]);
        a ^= 1;
        if (a == 0) aphase ^= 1;
      }
      if (!ok) break;
      const int row = tm * kOzM + quarter * 32 + lane;
      if (row < P.M) {
        const int ea = oz_exp(P.rmA[row]);
        double *crow = P.C + (size_t)row * P.ldc;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int cn = tn * kOzN + 16 * half + j;
          if (cn >= P.N) continue;
          // levels 0-3 and 4-6 as two exact 64-bit fixed-point integers (level l weighs
          // 2^{-8(l+2)}: hi in units of 2^-40, lo in units of 2^-64), then two conversions and
          // one FMA: the FP64 units of this GPU are slow, the integer ones are not
          const long long hi = ((long long)acc[0][j] << 24) + ((long long)acc[1][j] << 16) +
                               ((long long)acc[2][j] << 8) + (long long)acc[3][j];
          const long long lo = ((long long)acc[4][j] << 16) + ((long long)acc[5][j] << 8) + (long long)acc[6][j];
          const double v = fma((double)hi, 0x1p-40, (double)lo * 0x1p-64) * oz_pow2(ea + oz_exp(P.rmB[cn]));
          crow[cn] = (P.beta == 0.0) ? P.alpha * v : fma(P.alpha, v, P.beta * crow[cn]);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kOzAccCols);
  }
}

// ---------------------------------------------------------------------------------------
namespace {

int oz_pad(int x, int m) { return (x + m - 1) / m * m; }
size_t oz_align(size_t x) { return (x + 255) / 256 * 256; }
size_t oz_plane_bytes(int rows, int K) { return (size_t)kOzS * oz_pad(rows, 128) * oz_pad(K, kOzK) * 2; }

template <bool TRANS>
cudaError_t oz_split(const Launch &L, const double *src, int rows, int K, int ld, unsigned long long *rmax,
                     uint16_t *planes) {
  const int rows_pad = oz_pad(rows, 128), ldk = oz_pad(K, kOzK);
  cudaError_t e = cudaMemsetAsync(rmax, 0, (size_t)rows * sizeof(unsigned long long), L.stream);
  if (e != cudaSuccess) return e;
  k_oz_rowmax<TRANS><<<dim3((K + 63) / 64, (rows + 31) / 32), 256, 0, L.stream>>>(src, rows, K, ld, rmax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k_oz_slices<TRANS><<<dim3(ldk / 64, rows_pad / 32), 256, 0, L.stream>>>(src, rows, K, ld, rows_pad, ldk, rmax,
                                                                          planes);
  return cudaGetLastError();
}

}  // namespace

size_t gemm_oz_ws_bytes(int M, int N, int K) {
  return oz_align(oz_plane_bytes(M, K)) + oz_align(oz_plane_bytes(N, K)) + oz_align((size_t)M * 8) +
         oz_align((size_t)N * 8);
}

bool gemm_oz_ok(int M, int N, int K) { return M > 0 && N > 0 && K > 0 && K <= kOzMaxK; }

// C = alpha op(A) op(B) + beta C in FP64 (op(A): M x K, op(B): K x N; transA: A is K x M,
// transB: B is N x K), the products on the tensor cores; ws: gemm_oz_ws_bytes(M, N, K) bytes,
// 256-byte aligned.
cudaError_t launch_gemm_oz(const Launch &L, const double *A, int lda, bool transA, const double *B, int ldb,
                           bool transB, double *C, int ldc, int M, int N, int K, double alpha, double beta, void *ws) {
  if (!gemm_oz_ok(M, N, K) || !ws || !aligned16(ws)) return cudaErrorInvalidValue;
  uint8_t *p = static_cast<uint8_t *>(ws);
  uint16_t *pa = reinterpret_cast<uint16_t *>(p);
  p += oz_align(oz_plane_bytes(M, K));
  uint16_t *pb = reinterpret_cast<uint16_t *>(p);
  p += oz_align(oz_plane_bytes(N, K));
  unsigned long long *rmA = reinterpret_cast<unsigned long long *>(p);
  p += oz_align((size_t)M * 8);
  unsigned long long *rmB = reinterpret_cast<unsigned long long *>(p);
  cudaError_t e;
  e = transA ? oz_split<true>(L, A, M, K, lda, rmA, pa) : oz_split<false>(L, A, M, K, lda, rmA, pa);
  if (e != cudaSuccess) return e;
  // the rows of op(B)^T: B's rows when B is N x K, else its columns
  e = transB ? oz_split<false>(L, B, N, K, ldb, rmB, pb) : oz_split<true>(L, B, N, K, ldb, rmB, pb);
  if (e != cudaSuccess) return e;
  const int ldk = oz_pad(K, kOzK), rows_a = oz_pad(M, 128), rows_b = oz_pad(N, 128);
  const uint64_t nch = (uint64_t)(ldk / kOzK);
  CUtensorMap tmA, tmB;
  if (!plane_map(&tmA, pa, (uint64_t)kOzS * rows_a * nch, 128) ||
      !plane_map(&tmB, pb, (uint64_t)kOzS * rows_b * nch, (uint32_t)kOzN))
    return cudaErrorInvalidValue;
  OzParams P;
  std::memset(&P, 0, sizeof(P));
  P.M = M;
  P.N = N;
  P.K = K;
  P.tiles_m = (M + kOzM - 1) / kOzM;
  P.tiles_n = (N + kOzN - 1) / kOzN;
  P.nch = (int)nch;
  P.tiles_ra = rows_a / 128;
  P.tiles_rb = rows_b / 128;
  P.alpha = alpha;
  P.beta = beta;
  P.C = C;
  P.ldc = ldc;
  P.rmA = rmA;
  P.rmB = rmB;
  const int smem = kOzStages * kOzStageBytes + 1024;
  if ((e = ensure_dynamic_smem<k_gemm_oz>(smem)) != cudaSuccess) return e;
  const int ntiles = P.tiles_m * P.tiles_n;
  const int grid = ntiles < L.sms ? ntiles : L.sms;
  k_gemm_oz<<<grid, kOzThreads, smem, L.stream>>>(P, tmA, tmB, L.status);
  return cudaGetLastError();
}

}  // namespace gift
