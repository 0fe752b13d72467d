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
//   k_split_planes   FP32 or BF16 source (rows x K, or K x rows when transposed) -> `nt` BF16
//                    term planes, each rows_pad x ldk (zero padded to a multiple of 128 rows
//                    and 64 columns) and blocked: the 128-row x 64-K tile (r / 128, k / 64) is
//                    16 KB of consecutive memory, rows of 64 K-major elements.  A
//                    128-byte-swizzled TMA box of 64 x 128 (or 64 x 64) elements then reads one
//                    contiguous run from DRAM and lands as a K-major tcgen05 operand.
//   k_gemm_split     persistent over 128 x 128 tiles of C = alpha A B^T (A: M x K planes,
//                    B: N x K planes; N <= 64 takes 128 x 64 tiles).  Warp 8 streams each
//                    64-wide K chunk's term tiles with TMA (2 to 6 stages, as many as 220 KB of
//                    shared memory hold); warp 9 issues the products' 128 x N x 16 MMAs into
//                    one of four TMEM accumulators, a fresh one per chunk; warps 0-7 add the
//                    finished chunk into registers (32 rows x N / 2 columns each) and
//                    store alpha times the sum once the tile's last chunk is in.  A lower
//                    triangular operand (A: row i has k <= i; B: row j has k <= j) limits the
//                    tile's K range, so triangular factors cost half the MMAs.
// Every mbarrier wait is clock-bounded and reports GIFT_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include <cuda_bf16.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kGM = 128, kGK = 64;   // tile rows and K chunk; the tile's N (BN) is 128 or 64
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 32 * (kGEpiWarps + 2);
constexpr int kGTile = 128 * 128;              // bytes of one 128-row x 64-K BF16 term tile of A
constexpr long long kGWait = 4000000000LL;     // about two seconds of SM clock

constexpr int kGMaxProducts = 9;
constexpr int kGMaxStages = 6;
constexpr int kGSmemBudget = 220 * 1024;   // stage ring bytes

struct GemmTcParams {
  int M, N, K;
  int ldc;
  float alpha;
  int tiles_m, tiles_n, ntiles;   // ntiles counts work units: tiles (lower tiles only with
                                  // lower_tiles) times K slices
  int nta, ntb;            // term planes of A and B
  int tiles_ra, tiles_rb;  // 128-row tiles of one plane of A and of B
  int nch;                 // 64-wide K chunks of a plane row (ldk / 64)
  int nprod;               // products (pa[q], pb[q]) of the A and B terms, smallest first
  int8_t pa[kGMaxProducts], pb[kGMaxProducts];
  int a_lower, b_lower, lower_tiles;
  int ksplit, cps;         // K slices per tile and 64-wide chunks per slice
  size_t slice_stride;     // ksplit > 1: slice s of the result at C + s * slice_stride
  int stages, stage_bytes;
  float *C;
  const int *skip;         // nullable: the kernel does nothing while *skip != 0
};

// Work units are ranked heaviest first (with a lower-triangular B the last column blocks need
// the most K, with a lower-triangular A the last row blocks), and CTA b takes ranks b, 2G-1-b,
// 2G+b, 4G-1-b, ... of the G CTAs: a snake that pairs heavy units with light ones.  A unit is a
// 128 x 128 tile and one of its ksplit K slices.
__device__ __forceinline__ void gemm_tile_of(const GemmTcParams &P, int t, int &tm, int &tn, int &slice) {
  // (tiles_m, tiles_n count tiles of 128 rows and of the kernel's BN columns)
  slice = t % P.ksplit;
  t /= P.ksplit;
  if (P.lower_tiles) {   // tiles with tn <= tm, row by row
    int r = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while (r * (r + 1) / 2 > t) --r;
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    tm = r;
    tn = t - r * (r + 1) / 2;
  } else if (P.b_lower && !P.a_lower) {
    tn = P.tiles_n - 1 - t / P.tiles_m;
    tm = t % P.tiles_m;
  } else {
    tm = P.a_lower ? P.tiles_m - 1 - t / P.tiles_n : t / P.tiles_n;
    tn = t % P.tiles_n;
  }
}

// The i-th unit rank of CTA b (or -1 past the end).
__device__ __forceinline__ int gemm_rank(const GemmTcParams &P, int b, int i) {
  const int G = gridDim.x;
  const int r = (i & 1) ? (i + 1) * G - 1 - b : i * G + b;
  return r < P.ntiles ? r : -1;
}

// The unit's chunk range [c0, c1) of 64-wide K chunks.
template <int BN>
__device__ __forceinline__ void gemm_chunks(const GemmTcParams &P, int tm, int tn, int slice, int &c0, int &c1) {
  int kend = P.K;
  if (P.a_lower && (tm + 1) * kGM < kend) kend = (tm + 1) * kGM;
  if (P.b_lower && (tn + 1) * BN < kend) kend = (tn + 1) * BN;
  const int nch = (kend + kGK - 1) / kGK;
  c0 = slice * P.cps;
  c1 = c0 + P.cps < nch ? c0 + P.cps : nch;
  if (c1 < c0) c1 = c0;
}

}  // namespace

// 32 rows x 64 k of the planes per block of 256 threads; each thread splits 8 consecutive k.
// The source is FP32 or BF16 (a BF16 value is its own first term, the others are zero).
template <typename Src>
__device__ __forceinline__ float ld_src(const Src *p, size_t i) {
  if constexpr (sizeof(Src) == 2) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  else return p[i];
}

template <typename Src, bool TRANS>
__global__ void __launch_bounds__(256) k_split_planes(const Src *__restrict__ src, int rows, int K, int ld, int nt,
                                                      int rows_pad, int ldk, uint16_t *__restrict__ planes,
                                                      const int *skip) {
  __shared__ float tile[32][64 + 1];
  if (skip && *skip) return;
  const int r0 = blockIdx.y * 32, k0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  if (!TRANS) {
    for (int q = tid; q < 32 * 64; q += 256) {
      const int r = q >> 6, k = q & 63;
      const int gr = r0 + r, gk = k0 + k;
      tile[r][k] = (gr < rows && gk < K) ? ld_src(src, (size_t)gr * ld + gk) : 0.0f;
    }
  } else {
    for (int q = tid; q < 32 * 64; q += 256) {
      const int k = q >> 5, r = q & 31;   // source row k, column r: coalesced along r
      const int gr = r0 + r, gk = k0 + k;
      tile[r][k] = (gr < rows && gk < K) ? ld_src(src, (size_t)gk * ld + gr) : 0.0f;
    }
  }
  __syncthreads();
  const int r = tid >> 3, kb = (tid & 7) * 8;
  const int gr = r0 + r;
  if (gr >= rows_pad) return;
  uint32_t w1[4], w2[4], w3[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) tc::bf16_split3x2(tile[r][kb + 2 * q], tile[r][kb + 2 * q + 1], w1[q], w2[q], w3[q]);
  const size_t off = ((size_t)(gr >> 7) * (ldk >> 6) + (k0 >> 6)) * 8192 + (size_t)(gr & 127) * 64 + kb;
  const size_t plane = (size_t)rows_pad * ldk;
  *reinterpret_cast<uint4 *>(planes + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  if (nt > 1) *reinterpret_cast<uint4 *>(planes + plane + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  if (nt > 2) *reinterpret_cast<uint4 *>(planes + 2 * plane + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
}

// SB > 1 (A a single term): the products x y_0 .. x y_{SB-1} are one MMA per K step with the
// B term tiles stacked as N = SB x BN rows (they sit back to back in the stage), so A is read
// from shared memory once per K step instead of once per product; each product lands in its
// own BN-column group of the accumulator and the epilogue adds the groups, smallest first.
template <int BN, int SB>
__global__ void __launch_bounds__(kGThreads, 1) k_gemm_split(const __grid_constant__ GemmTcParams P,
                                                             const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB, int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  constexpr int NACC = (SB > 1) ? 2 : 4;       // TMEM accumulators (a fresh one per chunk)
  constexpr int ACOLS = SB * BN;                // columns of one accumulator
  constexpr uint32_t TCOLS = (NACC * ACOLS <= 256) ? 256u : 512u;
  static_assert(NACC * ACOLS <= 512 && ACOLS <= 256, "accumulators exceed tensor memory or the MMA's N");
  __shared__ uint64_t full[kGMaxStages], empty[kGMaxStages], afull[NACC], aempty[NACC];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (P.skip && *P.skip) return;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, TCOLS);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < P.stages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
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
      int s = 0, phase = 0;   // ring position; phase flips when s wraps
      long long g = 0;        // loads issued
      bool ok = true;
      for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0 && ok; ++i) {
        int tm, tn, sl, c0, c1;
        gemm_tile_of(P, t, tm, tn, sl);
        gemm_chunks<BN>(P, tm, tn, sl, c0, c1);
        for (int c = c0; c < c1; ++c) {
          if (!(ok = wait(&empty[s], (uint32_t)(phase ^ 1)))) break;
          uint8_t *st = sm + (size_t)s * P.stage_bytes;
          tc::mbar_arrive_expect_tx(&full[s], (uint32_t)P.stage_bytes);
          // blocked planes: the box of (plane p, row tile, chunk c) starts at row
          // ((p * tiles + tile) * nch + c) * 128 of the 64-wide view
          for (int p = 0; p < P.nta; ++p)
            tc::tma_load_2d(st + p * kGTile, &tmA, 0, ((p * P.tiles_ra + tm) * P.nch + c) * 128, &full[s]);
          const int tb = (tn * BN) >> 7, sub = (tn * BN) & 127;
          for (int p = 0; p < P.ntb; ++p)
            tc::tma_load_2d(st + P.nta * kGTile + p * (BN * 128), &tmB, 0, ((p * P.tiles_rb + tb) * P.nch + c) * 128 + sub,
                            &full[s]);
          ++g;
          if (++s == P.stages) {
            s = 0;
            phase ^= 1;
          }
        }
      }
      if (failed) {   // let this CTA's loads land before the shared memory is released
        for (int q = 0; q < P.stages; ++q) {
          const long long n = g / P.stages + (q < (int)(g % P.stages) ? 1 : 0);   // loads into stage q
          if (n) tc::mbar_wait_bounded(&full[q], (uint32_t)((n - 1) & 1), kGWait);
        }
      }
    }
  } else if (warp == kGEpiWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kGM, ACOLS);
      // the products' operand offsets, in registers (a dynamically indexed parameter array
      // would be copied to local memory)
      uint32_t offa[kGMaxProducts], offb[kGMaxProducts];
#pragma unroll
      for (int q = 0; q < kGMaxProducts; ++q) {
        offa[q] = (uint32_t)(P.pa[q] * kGTile);
        offb[q] = (uint32_t)(P.nta * kGTile + P.pb[q] * (BN * 128));
      }
      int s = 0, phase = 0, a = 0, aphase = 0;
      bool ok = true;
      for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0 && ok; ++i) {
        int tm, tn, sl, c0, c1;
        gemm_tile_of(P, t, tm, tn, sl);
        gemm_chunks<BN>(P, tm, tn, sl, c0, c1);
        for (int c = c0; c < c1; ++c) {
          if (!(ok = wait(&aempty[a], (uint32_t)(aphase ^ 1)))) break;
          if (!(ok = wait(&full[s], (uint32_t)phase))) break;
          tc::fence_after_sync();
          const uint32_t base = tc::smem_u32(sm + (size_t)s * P.stage_bytes);
          const uint32_t d = tmem + (uint32_t)(a * ACOLS);
          if (SB > 1) {   // A term 0 against the stacked B terms 0 .. SB-1
            const uint32_t bb = base + (uint32_t)(P.nta * kGTile);
#pragma unroll
            for (int k = 0; k < kGK / 16; ++k)
              tc::mma_bf16(d, tc::sdesc_kmajor_sw128(base + 32 * k), tc::sdesc_kmajor_sw128(bb + 32 * k), idesc,
                           k > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int q = 0; q < kGMaxProducts; ++q) {
            if (SB == 1 && q < P.nprod) {
              const uint32_t ab = base + offa[q], bb = base + offb[q];
#pragma unroll
              for (int k = 0; k < kGK / 16; ++k)
                tc::mma_bf16(d, tc::sdesc_kmajor_sw128(ab + 32 * k), tc::sdesc_kmajor_sw128(bb + 32 * k), idesc,
                             (q > 0 || k > 0) ? 1u : 0u);
            }
          }
          tc::mma_commit(&empty[s]);
          tc::mma_commit(&afull[a]);
          if (++s == P.stages) {
            s = 0;
            phase ^= 1;
          }
          if (++a == NACC) {
            a = 0;
            aphase ^= 1;
          }
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 0-7): 32 rows x BN / 2 columns each ----------------
    constexpr int NC = BN / 2;   // columns per warp
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int a = 0, aphase = 0;
    for (int i = 0, t; (t = gemm_rank(P, blockIdx.x, i)) >= 0; ++i) {
      int tm, tn, sl, c0, c1;
      gemm_tile_of(P, t, tm, tn, sl);
      gemm_chunks<BN>(P, tm, tn, sl, c0, c1);
      float acc[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) acc[i] = 0.0f;
      bool ok = true;
      // with N = 64, two chunks per round trip: both accumulators are read with one completion
      // wait, then added in chunk order (with N = 128 the registers hold one chunk)
      constexpr int CG = (BN == 64 && SB == 1) ? 2 : 1;
      if (SB > 1) {
        for (int c = c0; c < c1; ++c) {
          if (!(ok = wait(&afull[a], (uint32_t)aphase))) break;
          tc::fence_after_sync();
          uint32_t r[SB][NC];
#pragma unroll
          for (int gq = 0; gq < SB; ++gq)
#pragma unroll
            for (int g = 0; g < NC / 32; ++g)
              tc::tmem_ld32_nowait(tmem + lane_off + (uint32_t)(a * ACOLS + gq * BN + NC * half + 32 * g),
                                   r[gq] + 32 * g);
#pragma unroll
          for (int gq = 0; gq < SB; ++gq)
#pragma unroll
            for (int g = 0; g < NC / 32; ++g) tc::tmem_wait_ld(r[gq] + 32 * g);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&aempty[a]);
          if (++a == NACC) {
            a = 0;
            aphase ^= 1;
          }
#pragma unroll
          for (int i = 0; i < NC; ++i) {
            float sum = __uint_as_float(r[SB - 1][i]);
#pragma unroll
            for (int gq = SB - 2; gq >= 0; --gq) sum = __fadd_rn(sum, __uint_as_float(r[gq][i]));
            acc[i] = __fadd_rn(acc[i], sum);
          }
        }
      }
      for (int c = c0; c < c1 && SB == 1; c += CG) {
        const int n2 = (c1 - c) < CG ? (c1 - c) : CG;
        const int a1 = (a + 1 == NACC) ? 0 : a + 1;
        const int aphase1 = (a + 1 == NACC) ? (aphase ^ 1) : aphase;
        if (!(ok = wait(&afull[a], (uint32_t)aphase))) break;
        if (n2 == 2 && !(ok = wait(&afull[a1], (uint32_t)aphase1))) break;
        tc::fence_after_sync();
        uint32_t r[CG][NC];
        const uint32_t col = tmem + lane_off + (uint32_t)(a * ACOLS + NC * half);
        const uint32_t col1 = tmem + lane_off + (uint32_t)(a1 * ACOLS + NC * half);
#pragma unroll
        for (int g = 0; g < NC / 32; ++g) tc::tmem_ld32_nowait(col + 32 * g, r[0] + 32 * g);
        if (CG == 2 && n2 == 2) {
#pragma unroll
          for (int g = 0; g < NC / 32; ++g) tc::tmem_ld32_nowait(col1 + 32 * g, r[CG - 1] + 32 * g);
        }
#pragma unroll
        for (int g = 0; g < NC / 32; ++g) tc::tmem_wait_ld(r[0] + 32 * g);
        if (CG == 2 && n2 == 2) {
#pragma unroll
          for (int g = 0; g < NC / 32; ++g) tc::tmem_wait_ld(r[CG - 1] + 32 * g);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&aempty[a]);
          if (n2 == 2) tc::mbar_arrive(&aempty[a1]);
        }
        for (int u = 0; u < n2; ++u)
          if (++a == NACC) {
            a = 0;
            aphase ^= 1;
          }
#pragma unroll
        for (int i = 0; i < NC; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(r[0][i]));
        if (CG == 2 && n2 == 2) {
#pragma unroll
          for (int i = 0; i < NC; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(r[CG - 1][i]));
        }
      }
      if (!ok) break;
      const int row = tm * kGM + quarter * 32 + lane;
      const int col0 = tn * BN + half * NC;
      if (row < P.M) {
        float *crow = P.C + (size_t)sl * P.slice_stride + (size_t)row * P.ldc + col0;
        if (col0 + NC <= P.N && ((((uintptr_t)crow) & 15) == 0)) {
#pragma unroll
          for (int q = 0; q < NC / 4; ++q)
            reinterpret_cast<float4 *>(crow)[q] =
                make_float4(__fmul_rn(acc[4 * q], P.alpha), __fmul_rn(acc[4 * q + 1], P.alpha),
                            __fmul_rn(acc[4 * q + 2], P.alpha), __fmul_rn(acc[4 * q + 3], P.alpha));
        } else {
#pragma unroll
          for (int i = 0; i < NC; ++i)
            if (col0 + i < P.N) crow[i] = __fmul_rn(acc[i], P.alpha);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TCOLS);
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

}  // namespace

// Blocked BF16 planes viewed as rows of 64 elements (128 bytes): boxes of 64 x box_rows,
// 128-byte swizzle.  (Also used by the FP64-accurate GEMM.)
bool plane_map(CUtensorMap *m, const uint16_t *base, uint64_t rows_total, uint32_t box_rows) {
  auto enc = gemm_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kGK, rows_total};
  const cuuint64_t strides[1] = {(cuuint64_t)kGK * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kGK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

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

template <typename Src>
static cudaError_t split_planes_t(const Launch &L, const Src *src, int rows, int K, int ld, bool transpose, int nt,
                                  uint16_t *planes, const int *skip) {
  const int rows_pad = pad_to(rows, 128), ldk = pad_to(K, kGK);
  const dim3 grid(ldk / 64, rows_pad / 32);
  if (transpose)
    k_split_planes<Src, true><<<grid, 256, 0, L.stream>>>(src, rows, K, ld, nt, rows_pad, ldk, planes, skip);
  else
    k_split_planes<Src, false><<<grid, 256, 0, L.stream>>>(src, rows, K, ld, nt, rows_pad, ldk, planes, skip);
  return cudaGetLastError();
}

cudaError_t launch_split_planes(const Launch &L, const float *src, int rows, int K, int ld, bool transpose, int nt,
                                uint16_t *planes, const int *skip) {
  return split_planes_t<float>(L, src, rows, K, ld, transpose, nt, planes, skip);
}

cudaError_t launch_split_planes_bf16(const Launch &L, const void *src, int rows, int K, int ld, bool transpose,
                                     uint16_t *planes, const int *skip) {
  return split_planes_t<__nv_bfloat16>(L, static_cast<const __nv_bfloat16 *>(src), rows, K, ld, transpose, 1, planes,
                                       skip);
}

// Sum of the K slices in slice order (round-to-nearest FP32), times alpha.
__global__ void __launch_bounds__(256) k_sum_slices_tc(const float *__restrict__ parts, int ksplit, size_t stride,
                                                       int M, int N, int ld, float alpha, float *__restrict__ out,
                                                       int ldo, const int *skip) {
  if (skip && *skip) return;
  const size_t n = (size_t)M * N;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / N, c = i - r * N;
    float s = parts[r * ld + c];
    for (int k = 1; k < ksplit; ++k) s = __fadd_rn(s, parts[(size_t)k * stride + r * ld + c]);
    out[r * ldo + c] = __fmul_rn(s, alpha);
  }
}

cudaError_t launch_gemm_planes(const Launch &L, const GemmPlanes &g) {
  const int ldk = pad_to(g.K, kGK);
  const int rows_a = pad_to(g.M, 128), rows_b = pad_to(g.N, 128);
  if (g.nta < 1 || g.nta > 3 || g.ntb < 1 || g.ntb > 3 || g.ksplit < 1) return cudaErrorInvalidValue;
  if (g.lower_tiles && g.M != g.N) return cudaErrorInvalidValue;
  const int BN = (g.N <= 64 && !g.lower_tiles) ? 64 : 128;   // the tile's columns
  CUtensorMap tmA, tmB;
  const uint64_t nchl = (uint64_t)(ldk / kGK);
  if (!plane_map(&tmA, g.pa, (uint64_t)g.nta * rows_a * nchl, 128) ||
      !plane_map(&tmB, g.pb, (uint64_t)g.ntb * rows_b * nchl, (uint32_t)BN))
    return cudaErrorInvalidValue;
  GemmTcParams P;
  std::memset(&P, 0, sizeof(P));
  P.M = g.M;
  P.N = g.N;
  P.K = g.K;
  P.alpha = g.ksplit > 1 ? 1.0f : g.alpha;
  P.tiles_m = (g.M + kGM - 1) / kGM;
  P.tiles_n = (g.N + BN - 1) / BN;
  const int tiles = g.lower_tiles ? P.tiles_m * (P.tiles_m + 1) / 2 : P.tiles_m * P.tiles_n;
  P.ksplit = g.ksplit;
  const int nch = ldk / kGK;
  P.cps = (nch + g.ksplit - 1) / g.ksplit;
  P.ntiles = tiles * g.ksplit;
  P.nta = g.nta;
  P.ntb = g.ntb;
  P.tiles_ra = rows_a / 128;
  P.tiles_rb = rows_b / 128;
  P.nch = ldk / kGK;
  // the products x_i y_j kept: i + j <= 2 (0-based) at FP32 precision, i + j <= 1 otherwise;
  // smallest first
  const int maxsum = g.fp32 ? 2 : 1;
  for (int sum = maxsum; sum >= 0; --sum)
    for (int i = g.nta - 1; i >= 0; --i) {
      const int j = sum - i;
      if (j >= 0 && j < g.ntb) {
        P.pa[P.nprod] = (int8_t)i;
        P.pb[P.nprod] = (int8_t)j;
        ++P.nprod;
      }
    }
  P.a_lower = g.a_lower ? 1 : 0;
  P.b_lower = g.b_lower ? 1 : 0;
  P.lower_tiles = g.lower_tiles ? 1 : 0;
  P.stage_bytes = g.nta * kGTile + g.ntb * BN * 128;
  P.stages = kGSmemBudget / P.stage_bytes;
  if (P.stages > kGMaxStages) P.stages = kGMaxStages;
  if (P.stages < 2) return cudaErrorInvalidValue;
  P.skip = g.skip;
  float *dst = g.C;
  int ldc = g.ldc;
  if (g.ksplit > 1) {
    if (!g.parts) return cudaErrorInvalidValue;
    dst = g.parts;
    ldc = g.N;
    P.slice_stride = (size_t)g.M * g.N;
  }
  P.C = dst;
  P.ldc = ldc;
  const int smem = P.stages * P.stage_bytes + 1024;
  const int grid = P.ntiles < L.sms ? P.ntiles : L.sms;
  // a single A term: its products with B terms 0 .. nprod-1 as one stacked MMA per K step
  // (the products are (0, j), j < nprod, whenever nta == 1)
  const int sb = (g.nta == 1 && P.nprod > 1 && P.nprod * BN <= 256) ? P.nprod : 1;
  cudaError_t e;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e2 = ensure_dynamic_smem<decltype(kern)::value>(smem);
    if (e2 != cudaSuccess) return e2;
    decltype(kern)::value<<<grid, kGThreads, smem, L.stream>>>(P, tmA, tmB, L.status);
    return cudaGetLastError();
  };
  if (BN == 64) {
    if (sb == 3) e = go(std::integral_constant<decltype(&k_gemm_split<64, 3>), &k_gemm_split<64, 3>>{});
    else if (sb == 2) e = go(std::integral_constant<decltype(&k_gemm_split<64, 2>), &k_gemm_split<64, 2>>{});
    else e = go(std::integral_constant<decltype(&k_gemm_split<64, 1>), &k_gemm_split<64, 1>>{});
  } else {
    if (sb == 2) e = go(std::integral_constant<decltype(&k_gemm_split<128, 2>), &k_gemm_split<128, 2>>{});
    else e = go(std::integral_constant<decltype(&k_gemm_split<128, 1>), &k_gemm_split<128, 1>>{});
  }
  if (e != cudaSuccess || g.ksplit == 1) return e;
  const size_t n = (size_t)g.M * g.N;
  int sg = (int)((n + 255) / 256);
  if (sg > L.sms * 4) sg = L.sms * 4;
  k_sum_slices_tc<<<sg, 256, 0, L.stream>>>(g.parts, g.ksplit, P.slice_stride, g.M, g.N, g.N, g.alpha, g.C, g.ldc,
                                           g.skip);
  return cudaGetLastError();
}

size_t gemm_tc_parts_floats(int M, int N, int ksplit) { return ksplit > 1 ? (size_t)ksplit * M * N : 0; }

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
  GemmPlanes q;
  q.pa = pa;
  q.pb = pb;
  q.M = g.M;
  q.N = g.N;
  q.K = g.K;
  q.nta = q.ntb = nt;
  q.fp32 = nt == 3;
  q.a_lower = g.a_lower;
  q.b_lower = g.b_lower_t;
  q.alpha = g.alpha;
  q.C = g.C;
  q.ldc = g.ldc;
  return launch_gemm_planes(L, q);
}

}  // namespace gift
