// FP32 GEMMs on the 5th-generation tensor cores with exact BF16 operand splits.
//
// The full-rank transforms of the GIFT reading notes (core idea step 3, eq. (11): W~ = L_G^-1 W
// L_A^-T; simplification 1, eq. (16): W~ = W L_A^-T; eq. (14): the map back W^ = L_G X L_A^T)
// and the sketch of the factor refresh (simplification 2, eq. (17)) are dense FP32
// contractions.  They run here on tcgen05 (kind::f16, BF16 operands, FP32 accumulation).
//
// Precision.  Every FP32 operand x is split into BF16 terms x = x1 + x2 + x3 (tc.cuh,
// bf16_split3: exact).  A product of two BF16 terms is exact in FP32.  The FP32 precision sums
// the six products x_i y_j with i + j <= 4 (what is dropped is below 2^-23 |x||y| per product);
// the TC precision keeps two terms of each operand and three products (i + j <= 3, below
// 2^-15).  The tensor core's FP32 accumulation is not round to nearest, so one accumulator
// never sums more than one 64-wide K chunk (24 MMAs at FP32 precision): the epilogue warps add
// every chunk's accumulator into FP32 registers with round-to-nearest additions.
//
//   k_split_planes   FP32 source (rows x K, or K x rows when transposed) -> `nt` BF16 term
//                    planes, each rows_pad x ldk (K-major rows, zero padded to a multiple of
//                    128 rows and 64 columns), the layout a 128-byte-swizzled TMA box of
//                    64 x 128 elements reads as a K-major tcgen05 operand.
//   k_gemm_split     persistent over 128 x 128 tiles of C = alpha A B^T (A: M x K planes,
//                    B: N x K planes).  Warp 8 streams each 64-wide K chunk's term tiles with
//                    TMA (2 or 3 stages); warp 9 issues the products' 128 x 128 x 16 MMAs into
//                    one of two 128-column TMEM accumulators, a fresh one per chunk; warps 0-7
//                    add the finished chunk into registers (32 rows x 64 columns each) and
//                    store alpha times the sum once the tile's last chunk is in.  A lower
//                    triangular operand (A: row i has k <= i; B: row j has k <= j) limits the
//                    tile's K range, so triangular factors cost half the MMAs.
// Every mbarrier wait is clock-bounded and reports GIFT_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kGM = 128, kGN = 128, kGK = 64;
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 32 * (kGEpiWarps + 2);
constexpr int kGTile = 128 * 128;              // bytes of one 128-row x 64-K BF16 term tile
constexpr long long kGWait = 4000000000LL;     // about two seconds of SM clock

struct GemmTcParams {
  int M, N, K;
  int ldc;
  float alpha;
  int tiles_m, tiles_n, ntiles;
  int nta, ntb;            // term planes of A and B
  int rows_a, rows_b;      // padded rows of one plane (multiples of 128)
  int products;            // 3 (TC) or 6 (FP32)
  int a_lower, b_lower;
  int stages, stage_bytes;
  float *C;
};

// Tiles are ranked heaviest first (with a lower-triangular B the last column blocks need the
// most K, with a lower-triangular A the last row blocks), and CTA b takes ranks b, 2G-1-b,
// 2G+b, 4G-1-b, ... of the G CTAs: a snake that pairs heavy tiles with light ones.
__device__ __forceinline__ void gemm_tile_of(const GemmTcParams &P, int t, int &tm, int &tn) {
  if (P.b_lower && !P.a_lower) {
    tn = P.tiles_n - 1 - t / P.tiles_m;
    tm = t % P.tiles_m;
  } else {
    tm = P.a_lower ? P.tiles_m - 1 - t / P.tiles_n : t / P.tiles_n;
    tn = t % P.tiles_n;
  }
}

// The i-th tile rank of CTA b (or -1 past the end).
__device__ __forceinline__ int gemm_rank(const GemmTcParams &P, int b, int i) {
  const int G = gridDim.x;
  const int r = (i & 1) ? (i + 1) * G - 1 - b : i * G + b;
  return r < P.ntiles ? r : -1;
}

__device__ __forceinline__ int gemm_chunks(const GemmTcParams &P, int tm, int tn) {
  int kend = P.K;
  if (P.a_lower && (tm + 1) * kGM < kend) kend = (tm + 1) * kGM;
  if (P.b_lower && (tn + 1) * kGN < kend) kend = (tn + 1) * kGN;
  return (kend + kGK - 1) / kGK;
}

}  // namespace

// 32 rows x 64 k of the planes per block of 256 threads; each thread splits 8 consecutive k.
template <bool TRANS>
__global__ void __launch_bounds__(256) k_split_planes(const float *__restrict__ src, int rows, int K, int ld, int nt,
                                                      int rows_pad, int ldk, uint16_t *__restrict__ planes) {
  __shared__ float tile[32][64 + 1];
  const int r0 = blockIdx.y * 32, k0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  if (!TRANS) {
    for (int q = tid; q < 32 * 64; q += 256) {
      const int r = q >> 6, k = q & 63;
      const int gr = r0 + r, gk = k0 + k;
      tile[r][k] = (gr < rows && gk < K) ? src[(size_t)gr * ld + gk] : 0.0f;
    }
  } else {
    for (int q = tid; q < 32 * 64; q += 256) {
      const int k = q >> 5, r = q & 31;   // source row k, column r: coalesced along r
      const int gr = r0 + r, gk = k0 + k;
      tile[r][k] = (gr < rows && gk < K) ? src[(size_t)gk * ld + gr] : 0.0f;
    }
  }
  __syncthreads();
  const int r = tid >> 3, kb = (tid & 7) * 8;
  const int gr = r0 + r;
  if (gr >= rows_pad) return;
  uint32_t w1[4], w2[4], w3[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) tc::bf16_split3x2(tile[r][kb + 2 * q], tile[r][kb + 2 * q + 1], w1[q], w2[q], w3[q]);
  const size_t off = (size_t)gr * ldk + k0 + kb;
  const size_t plane = (size_t)rows_pad * ldk;
  *reinterpret_cast<uint4 *>(planes + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  if (nt > 1) *reinterpret_cast<uint4 *>(planes + plane + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  if (nt > 2) *reinterpret_cast<uint4 *>(planes + 2 * plane + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
}

__global__ void __launch_bounds__(kGThreads, 1) k_gemm_split(const __grid_constant__ GemmTcParams P,
                                                             const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB, int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[3], empty[3], afull[2], aempty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 256);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < P.stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&afull[a], 1);
      tc::mbar_init(&aempty[a], kGEpiWarps);
    }
    tc::fence_mbar_init();
    failed = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (failed) return false;
    if (!tc::mbar_wait_bounded(bar, parity, kGWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kGEpiWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tensormap(&tmA);
      tc::prefetch_tensormap(&tmB);
      long long g = 0;
      int issued[3] = {0, 0, 0};
      bool ok = true;
      for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0 && ok; ++i) {
        int tm, tn;
        gemm_tile_of(P, t, tm, tn);
        const int nch = gemm_chunks(P, tm, tn);
        for (int c = 0; c < nch; ++c, ++g) {
          const int s = (int)(g % P.stages);
          if (!(ok = wait(&empty[s], (uint32_t)(((g / P.stages) & 1) ^ 1)))) break;
          uint8_t *st = sm + (size_t)s * P.stage_bytes;
          tc::mbar_arrive_expect_tx(&full[s], (uint32_t)P.stage_bytes);
          for (int p = 0; p < P.nta; ++p)
            tc::tma_load_2d(st + p * kGTile, &tmA, c * kGK, p * P.rows_a + tm * kGM, &full[s]);
          for (int p = 0; p < P.ntb; ++p)
            tc::tma_load_2d(st + (P.nta + p) * kGTile, &tmB, c * kGK, p * P.rows_b + tn * kGN, &full[s]);
          ++issued[s];
        }
      }
      if (failed) {   // let this CTA's loads land before the shared memory is released
        for (int s = 0; s < P.stages; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&full[s], (uint32_t)((issued[s] - 1) & 1), kGWait);
      }
    }
  } else if (warp == kGEpiWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kGM, kGN);
      // products (i, j) of the A and B terms, smallest first
      const int pa6[6] = {2, 1, 0, 1, 0, 0}, pb6[6] = {0, 1, 2, 0, 1, 0};
      const int pa3[3] = {1, 0, 0}, pb3[3] = {0, 1, 0};
      const int *pa = P.products == 6 ? pa6 : pa3, *pb = P.products == 6 ? pb6 : pb3;
      long long g = 0, ch = 0;
      bool ok = true;
      for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0 && ok; ++i) {
        int tm, tn;
        gemm_tile_of(P, t, tm, tn);
        const int nch = gemm_chunks(P, tm, tn);
        for (int c = 0; c < nch; ++c, ++g, ++ch) {
          const int a = (int)(ch & 1);
          if (!(ok = wait(&aempty[a], (uint32_t)(((ch >> 1) & 1) ^ 1)))) break;
          const int s = (int)(g % P.stages);
          if (!(ok = wait(&full[s], (uint32_t)((g / P.stages) & 1)))) break;
          tc::fence_after_sync();
          const uint32_t base = tc::smem_u32(sm + (size_t)s * P.stage_bytes);
          const uint32_t d = tmem + (uint32_t)(a * kGN);
          bool first = true;
#pragma unroll 1
          for (int q = 0; q < P.products; ++q) {
            const uint32_t ab = base + pa[q] * kGTile, bb = base + (P.nta + pb[q]) * kGTile;
#pragma unroll
            for (int k = 0; k < kGK / 16; ++k) {
              tc::mma_bf16(d, tc::sdesc_kmajor_sw128(ab + 32 * k), tc::sdesc_kmajor_sw128(bb + 32 * k), idesc,
                           first ? 0u : 1u);
              first = false;
            }
          }
          tc::mma_commit(&empty[s]);
          tc::mma_commit(&afull[a]);
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 0-7): 32 rows x 64 columns each ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    long long ch = 0;
    for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0; ++i) {
      int tm, tn;
      gemm_tile_of(P, t, tm, tn);
      const int nch = gemm_chunks(P, tm, tn);
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      bool ok = true;
      for (int c = 0; c < nch; ++c, ++ch) {
        const int a = (int)(ch & 1);
        if (!(ok = wait(&afull[a], (uint32_t)((ch >> 1) & 1)))) break;
        tc::fence_after_sync();
        uint32_t r0[32], r1[32];
        const uint32_t col = tmem + lane_off + (uint32_t)(a * kGN + 64 * half);
        tc::tmem_ld32_nowait(col, r0);
        tc::tmem_ld32_nowait(col + 32, r1);
        tc::tmem_wait_ld(r0);
        tc::tmem_wait_ld(r1);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&aempty[a]);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc[i] = __fadd_rn(acc[i], __uint_as_float(r0[i]));
          acc[32 + i] = __fadd_rn(acc[32 + i], __uint_as_float(r1[i]));
        }
      }
      if (!ok) break;
      const int row = tm * kGM + quarter * 32 + lane;
      const int col0 = tn * kGN + half * 64;
      if (row < P.M) {
        float *crow = P.C + (size_t)row * P.ldc + col0;
        if (col0 + 64 <= P.N && ((((uintptr_t)crow) & 15) == 0)) {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            reinterpret_cast<float4 *>(crow)[q] =
                make_float4(__fmul_rn(acc[4 * q], P.alpha), __fmul_rn(acc[4 * q + 1], P.alpha),
                            __fmul_rn(acc[4 * q + 2], P.alpha), __fmul_rn(acc[4 * q + 3], P.alpha));
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (col0 + i < P.N) crow[i] = __fmul_rn(acc[i], P.alpha);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 gemm_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// BF16 planes [rows_total][ldk], boxes of 64 columns x 128 rows, 128-byte swizzle.
bool plane_map(CUtensorMap *m, const uint16_t *base, uint64_t rows_total, uint64_t ldk) {
  auto enc = gemm_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {ldk, rows_total};
  const cuuint64_t strides[1] = {ldk * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kGK, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pad_to(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

size_t gemm_tc_plane_bytes(int rows, int K, int nterms) {
  return (size_t)nterms * pad_to(rows, 128) * pad_to(K, kGK) * 2;
}

size_t gemm_tc_ws_bytes(int M, int N, int K, int nterms) {
  // A planes, then B planes, each 256-byte aligned
  return (gemm_tc_plane_bytes(M, K, nterms) + 255) / 256 * 256 + gemm_tc_plane_bytes(N, K, nterms);
}

bool gemm_tc_ok(const GemmArgs &g, const void *ws) {
  return !g.a_bf16 && !g.b_bf16 && !g.transA && !g.lower_tiles && g.M > 0 && g.N > 0 && g.K > 0 && ws &&
         aligned16(ws) && gemm_encoder() != nullptr;
}

cudaError_t launch_split_planes(const Launch &L, const float *src, int rows, int K, int ld, bool transpose, int nt,
                                uint16_t *planes) {
  const int rows_pad = pad_to(rows, 128), ldk = pad_to(K, kGK);
  const dim3 grid(ldk / 64, rows_pad / 32);
  if (transpose)
    k_split_planes<true><<<grid, 256, 0, L.stream>>>(src, rows, K, ld, nt, rows_pad, ldk, planes);
  else
    k_split_planes<false><<<grid, 256, 0, L.stream>>>(src, rows, K, ld, nt, rows_pad, ldk, planes);
  return cudaGetLastError();
}

cudaError_t launch_gemm_planes(const Launch &L, const uint16_t *pa, const uint16_t *pb, int M, int N, int K, int nt,
                               bool a_lower, bool b_lower, float alpha, float *C, int ldc) {
  const int rows_a = pad_to(M, 128), rows_b = pad_to(N, 128), ldk = pad_to(K, kGK);
  CUtensorMap tmA, tmB;
  if (!plane_map(&tmA, pa, (uint64_t)nt * rows_a, (uint64_t)ldk) ||
      !plane_map(&tmB, pb, (uint64_t)nt * rows_b, (uint64_t)ldk))
    return cudaErrorInvalidValue;
  GemmTcParams P;
  P.M = M;
  P.N = N;
  P.K = K;
  P.ldc = ldc;
  P.alpha = alpha;
  P.tiles_m = (M + kGM - 1) / kGM;
  P.tiles_n = (N + kGN - 1) / kGN;
  P.ntiles = P.tiles_m * P.tiles_n;
  P.nta = nt;
  P.ntb = nt;
  P.rows_a = rows_a;
  P.rows_b = rows_b;
  P.products = nt == 3 ? 6 : 3;
  P.a_lower = a_lower ? 1 : 0;
  P.b_lower = b_lower ? 1 : 0;
  P.stage_bytes = 2 * nt * kGTile;
  P.stages = nt == 3 ? 2 : 3;
  P.C = C;
  const int smem = P.stages * P.stage_bytes + 1024;
  cudaError_t e = ensure_dynamic_smem<k_gemm_split>(smem);
  if (e != cudaSuccess) return e;
  const int grid = P.ntiles < L.sms ? P.ntiles : L.sms;
  k_gemm_split<<<grid, kGThreads, smem, L.stream>>>(P, tmA, tmB, L.status);
  return cudaGetLastError();
}

// C = alpha op(A) op(B) with GemmArgs' conventions (FP32 operands, no transA), the operands
// split into `nt` BF16 term planes in ws (gemm_tc_ws_bytes(M, N, K, nt) bytes).
cudaError_t launch_gemm_tc(const Launch &L, const GemmArgs &g, int nt, void *ws) {
  uint16_t *pa = static_cast<uint16_t *>(ws);
  uint16_t *pb = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) +
                                              (gemm_tc_plane_bytes(g.M, g.K, nt) + 255) / 256 * 256);
  cudaError_t e = launch_split_planes(L, static_cast<const float *>(g.A), g.M, g.K, g.lda, false, nt, pa);
  if (e != cudaSuccess) return e;
  // B planes are N rows of K: B itself when transposed (N x K), else its transpose
  e = launch_split_planes(L, static_cast<const float *>(g.B), g.N, g.K, g.ldb, !g.transB, nt, pb);
  if (e != cudaSuccess) return e;
  return launch_gemm_planes(L, pa, pb, g.M, g.N, g.K, nt, g.a_lower, g.b_lower_t, g.alpha, g.C, g.ldc);
}

}  // namespace gift
