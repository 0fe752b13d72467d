// Rank-r projection P = X U on the 5th-generation tensor cores, split over K, with the
// coefficient finalize (Pc = P diag(c), its BF16 term planes) fused in after a grid-wide
// barrier.
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17): the whitened gradient
// is W~ = sigma^-1/2 W + ((W U) diag(c)) U^T, c = mu^-1/2 - sigma^-1/2; the map back uses
// c = mu^1/2 - sigma^1/2.  P = W U is a dense contraction over d_in (K), N = 32 outputs.
//
// Exactness: X and U are split exactly into BF16 terms (tc.cuh) and the products x_i u_j
// with i + j <= 4 (1-based; six of them) are accumulated in FP32 in tensor memory, which
// drops less than 2^-23 of each |x_k u_k|; the TC path keeps the three with i + j <= 3.
//
// CTA (row block rb, K slice sp): 128 rows of X against ktiles/nsplit K tiles of 64.
// Warp 8 streams each X tile (two 128 x 32 FP32 boxes) and the U^T term planes of that K
// range (32 x 64 BF16 boxes) through four shared-memory stages; warps 0-7 split the X tile
// into BF16 terms and store them to tensor memory (double-buffered A operand, one thread per
// row and 32 K values); warp 9 issues the MMAs with A from tensor memory and B = U^T from
// shared memory into a 128 x 32 FP32 accumulator per K tile (double-buffered), which the
// splitter warps add up in registers with round-to-nearest FP32.  The partial P of the slice goes to
// global memory; after one grid-wide barrier (the launch is cooperative when there is more
// than one slice, so all CTAs are resident; the wait is clock-bounded) each CTA sums its share
// of its row block's rows over the slices in slice order with a compensated FP32 sum, scales
// by c in FP64 and writes Pc and its term planes.  Every mbarrier wait is clock-bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kPM = 128;              // rows of X per CTA (TMEM lanes)
constexpr int kPK = 64;               // K per stage
constexpr int kPStages = 4;
constexpr int kPSplitWarps = 8;
constexpr int kPThreads = 32 * (kPSplitWarps + 2);
constexpr int kPXBox = 128 * 128;     // 128 rows x 32 FP32
constexpr int kPUBox = 32 * 128;      // 32 rows x 64 BF16
constexpr uint32_t kPTmemCols = 256;
constexpr uint32_t kPAcc = 0;         // two per-tile accumulators of 32 columns
constexpr uint32_t kPABuf = 64;       // two A buffers of 3 terms x 32 columns
constexpr long long kPWait = 4000000000LL;

struct ProjParams {
  const float *mu, *sigma;
  int rank, d_out, d_in;
  bool inverse;
  int nsplit, ktiles;
  float *part;             // nsplit x d_out x 32 slice partials
  float *Pc;               // d_out x 32
  uint16_t *pc_planes;     // term planes of Pc for the apply (pc_nplanes planes of d_out x 64 BF16)
  int pc_nplanes;
  unsigned int *counters;  // counters[0]: grid-barrier word, zero on entry
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <int NT>
struct PLayout {
  static constexpr int stage_bytes = 2 * kPXBox + NT * kPUBox;
  static constexpr int total = kPStages * stage_bytes;
};

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kPThreads, 1) k_lr_proj_tc(const __grid_constant__ ProjParams P,
                                                             const __grid_constant__ CUtensorMap tmX,
                                                             const __grid_constant__ CUtensorMap tmUT, int *status) {
  using Lay = PLayout<NT>;
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_full[kPStages], bar_empty[kPStages], bar_afull[2], bar_aempty[2], bar_cfull[2], bar_cempty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;
  __shared__ double coef[32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x / P.nsplit, sp = blockIdx.x - rb * P.nsplit;
  const int kt0 = (int)(((long long)P.ktiles * sp) / P.nsplit);
  const int kt1 = (int)(((long long)P.ktiles * (sp + 1)) / P.nsplit);
  const int r0 = rb * kPM;
  const int d_out = P.d_out;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, kPTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kPStages; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], kPSplitWarps + 1);   // the splitters read X, the MMAs read U^T
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar_afull[b], kPSplitWarps);
      tc::mbar_init(&bar_aempty[b], 1);
      tc::mbar_init(&bar_cfull[b], 1);
      tc::mbar_init(&bar_cempty[b], kPSplitWarps);
    }
    tc::fence_mbar_init();
    failed = 0;
  }
  if (warp == 1) {   // FP64 coefficients of the finalize, off the critical path
    const int k = lane;
    double c = 0.0;
    if (k < P.rank) {
      const double m = (double)P.mu[k], sg = (double)P.sigma[0];
      if (!(m > 0.0) || !(sg > 0.0)) {
        if (blockIdx.x == 0) set_status(status, GIFT_ERR_NOT_PD);
      } else {
        c = P.inverse ? (sqrt(m) - sqrt(sg)) : (1.0 / sqrt(m) - 1.0 / sqrt(sg));
      }
    }
    coef[k] = c;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (failed) return false;
    if (!tc::mbar_wait_bounded(bar, parity, kPWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kPSplitWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued[kPStages] = {};
      for (int kt = kt0, i = 0; kt < kt1; ++kt, ++i) {
        const int s = i % kPStages;
        if (!wait(&bar_empty[s], ((i / kPStages) & 1) ^ 1)) break;
        uint8_t *st = sm + s * Lay::stage_bytes;
        const int kx = kt * kPK;
        tc::mbar_arrive_expect_tx(&bar_full[s], Lay::stage_bytes);
        tc::tma_load_2d(st, &tmX, kx, r0, &bar_full[s]);
        tc::tma_load_2d(st + kPXBox, &tmX, kx + 32, r0, &bar_full[s]);
#pragma unroll
        for (int t = 0; t < NT; ++t) tc::tma_load_2d(st + 2 * kPXBox + t * kPUBox, &tmUT, kx, 32 * t, &bar_full[s]);
        ++issued[s];
      }
      if (failed) {
        for (int s = 0; s < kPStages; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&bar_full[s], (uint32_t)((issued[s] - 1) & 1), kPWait);
      }
    }
  } else if (warp == kPSplitWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kPM, 32);
      constexpr int np = (NT == 2) ? 3 : 6;
      constexpr int pa[6] = {NT == 2 ? 1 : 2, NT == 2 ? 0 : 1, 0, 1, 0, 0};
      constexpr int pb[6] = {0, 1, NT == 2 ? 0 : 2, 0, 1, 0};
      for (int kt = kt0, i = 0; kt < kt1; ++kt, ++i) {
        const int s = i % kPStages, b = i & 1;
        if (!wait(&bar_full[s], (uint32_t)((i / kPStages) & 1))) break;
        if (!wait(&bar_afull[b], (uint32_t)((i >> 1) & 1))) break;
        if (!wait(&bar_cempty[b], (uint32_t)(((i >> 1) & 1) ^ 1))) break;
        tc::fence_after_sync();
        const uint32_t ub = tc::smem_u32(sm + s * Lay::stage_bytes + 2 * kPXBox);
        // a fresh accumulator per K tile: the tensor core's FP32 accumulation is not rounded
        // to nearest, so it only sums one tile (the large x1 u1 product last); the tiles are
        // added in FP32 with round to nearest by the splitter warps
        uint32_t acc = 0;
#pragma unroll
        for (int p = 0; p < np; ++p) {
#pragma unroll
          for (int k = 0; k < kPK / 16; ++k) {
            tc::mma_bf16_ta(tmem + kPAcc + 32 * b, tmem + kPABuf + 96 * b + 32 * pa[p] + 8 * k,
                            tc::sdesc_kmajor_sw128(ub + pb[p] * kPUBox + 32 * k), idesc, acc);
            acc = 1;
          }
        }
        tc::mma_commit(&bar_empty[s]);    // U^T of this stage has been read
        tc::mma_commit(&bar_aempty[b]);   // A buffer b may be rewritten
        tc::mma_commit(&bar_cfull[b]);    // tile result ready
      }
    }
  } else {
    // ---------------- splitters (warps 0-7): thread = row, 32 K values per tile ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const int lr = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float accp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) accp[j] = 0.0f;
    // add the result of tile j (accumulator j & 1) into accp and hand the accumulator back
    auto fold = [&](int j) {
      const int c = j & 1;
      wait(&bar_cfull[c], (uint32_t)((j >> 1) & 1));
      tc::fence_after_sync();
      uint32_t raw[16];
      tc::tmem_ld16_nowait(tmem + lane_off + kPAcc + 32 * c + 16 * half, raw);
      tc::tmem_wait_ld16(raw);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_cempty[c]);
#pragma unroll
      for (int q = 0; q < 16; ++q) accp[q] = __fadd_rn(accp[q], __uint_as_float(raw[q]));
    };
    for (int kt = kt0, i = 0; kt < kt1; ++kt, ++i) {
      const int s = i % kPStages, b = i & 1;
      wait(&bar_full[s], (uint32_t)((i / kPStages) & 1));
      wait(&bar_aempty[b], (uint32_t)(((i >> 1) & 1) ^ 1));
      tc::fence_after_sync();
      const uint8_t *box = sm + s * Lay::stage_bytes + half * kPXBox;
      uint32_t w1[16], w2[16], w3[16];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = *reinterpret_cast<const float4 *>(box + ((lr * 128) + ((c ^ (lr & 7)) << 4)));
        tc::bf16_split3x2(x.x, x.y, w1[2 * c], w2[2 * c], w3[2 * c]);
        tc::bf16_split3x2(x.z, x.w, w1[2 * c + 1], w2[2 * c + 1], w3[2 * c + 1]);
      }
      const uint32_t abase = tmem + lane_off + kPABuf + 96 * b + 16 * half;
      tc::tmem_st16(abase, w1);
      tc::tmem_st16(abase + 32, w2);
      if (NT == 3) tc::tmem_st16(abase + 64, w3);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();   // X was read through the generic proxy; the refill is TMA
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&bar_afull[b]);
        tc::mbar_arrive(&bar_empty[s]);
      }
      if (i > 0) fold(i - 1);   // the MMAs of tile i can run meanwhile
    }
    if (kt1 > kt0) fold(kt1 - kt0 - 1);
    // slice partial of P: row lr, outputs 16 half .. 16 half + 15
    const float *v = accp;
    const int row = r0 + lr;
    if (row < d_out) {
      float4 *dst = reinterpret_cast<float4 *>(P.part + ((size_t)sp * d_out + row) * 32 + 16 * half);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    // ---- Pc = diag(c) (sum of the slices), and its term planes ----
    __threadfence();
    tc::named_bar_sync(1, 32 * kPSplitWarps);
    if (P.nsplit > 1 && tid == 0) {
      // grid-wide barrier (cooperative launch: every CTA is resident): all slices written
      atomicAdd(P.counters, 1u);
      const long long t0 = clock64();
      while (ld_acquire_u32(P.counters) < gridDim.x) {
        if (clock64() - t0 > kPWait) {
          set_status(status, GIFT_ERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    tc::named_bar_sync(1, 32 * kPSplitWarps);
    // this CTA's share of its row block; item = (row, 4 consecutive outputs).  The slices are
    // read sixteen at a time (independent L2 loads in flight) and added in slice order with a
    // compensated FP32 sum; the product with c is taken in FP64.
    const int ra = r0 + (kPM * sp) / P.nsplit, rz = r0 + (kPM * (sp + 1)) / P.nsplit;
    for (int item = tid; item < (rz - ra) * 8; item += 32 * kPSplitWarps) {
      const int rr = ra + (item >> 3), kb = 4 * (item & 7);
      if (rr >= d_out) continue;
      float sum[4] = {0.f, 0.f, 0.f, 0.f}, comp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q0 = 0; q0 < P.nsplit; q0 += 16) {
        float4 x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (q0 + u < P.nsplit)
            x[u] = __ldcg(reinterpret_cast<const float4 *>(P.part + ((size_t)(q0 + u) * d_out + rr) * 32 + kb));
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (q0 + u < P.nsplit) {
            const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float y = __fsub_rn(xs[e], comp[e]);
              const float t = __fadd_rn(sum[e], y);
              comp[e] = __fsub_rn(__fsub_rn(t, sum[e]), y);
              sum[e] = t;
            }
          }
      }
      float pc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pc[e] = (float)(coef[kb + e] * ((double)sum[e] - (double)comp[e]));
      *reinterpret_cast<float4 *>(P.Pc + (size_t)rr * 32 + kb) = make_float4(pc[0], pc[1], pc[2], pc[3]);
      if (P.pc_planes)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          tc::write_term_planes(P.pc_planes, (size_t)d_out, (size_t)rr, kb + e, pc[e], P.pc_nplanes);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kPTmemCols);
  }
}

// U term planes in both layouts the tensor-core kernels read, and the row-block counters of
// the projection set to zero: apply planes (rows of U, tc.cuh layout) and, for the
// projection, U^T planes: plane t row n = term t of U[:, n] (d_in BF16).  One CTA per 32 rows
// of U; the U^T planes are written through a shared-memory transpose so both layouts are
// stored in contiguous runs.
__global__ void __launch_bounds__(256) k_split_u(const float *__restrict__ U, int d_in, int rank, int nplanes_apply,
                                                 uint16_t *__restrict__ u_planes, uint16_t *__restrict__ ut_planes,
                                                 unsigned int *__restrict__ counters, int ncounters) {
  __shared__ uint16_t tr[3][32][34];   // [term][k][row in block], padded
  const int j0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 8 warps
  for (int jj = ty; jj < 32; jj += 8) {
    const int j = j0 + jj;
    const float x = (j < d_in && tx < rank) ? U[(size_t)j * rank + tx] : 0.0f;
    uint16_t t1, t2, t3;
    tc::bf16_split3(x, t1, t2, t3);
    if (j < d_in) {
      uint16_t *p0 = u_planes + (size_t)j * 64;
      p0[tx] = t1;
      p0[32 + tx] = t2;
      if (nplanes_apply > 1) {
        uint16_t *p1 = u_planes + (size_t)d_in * 64 + (size_t)j * 64;
        p1[tx] = t3;
        p1[32 + tx] = 0;
      }
    }
    tr[0][tx][jj] = t1;
    tr[1][tx][jj] = t2;
    tr[2][tx][jj] = t3;
  }
  __syncthreads();
  for (int r = ty; r < 96; r += 8) {   // plane row (term, k) = r: 32 consecutive j
    const int t = r >> 5, k = r & 31, j = j0 + tx;
    if (j < d_in) ut_planes[(size_t)r * d_in + j] = tr[t][k][tx];
  }
  if (blockIdx.x == 0)
    for (int c = threadIdx.x; c < ncounters; c += blockDim.x) counters[c] = 0u;
}

// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 proj_encoder() {
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

bool map2d(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t rows, uint64_t cols,
           uint32_t box_cols, uint32_t box_rows) {
  auto enc = proj_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int lr_proj_tc_splits(int sms, int d_out, int d_in) {
  const int tiles_m = (d_out + kPM - 1) / kPM;
  const int ktiles = (d_in + kPK - 1) / kPK;
  int ns = sms / tiles_m;
  if (ns < 1) ns = 1;
  if (ns > ktiles) ns = ktiles;
  return ns;
}

LrPlanes lr_planes(float *split, int d_out, int d_in) {
  LrPlanes p;
  p.pc = reinterpret_cast<uint16_t *>(split);
  p.u = reinterpret_cast<uint16_t *>(split + (size_t)64 * d_out);
  p.ut = reinterpret_cast<uint16_t *>(split + (size_t)64 * (d_out + d_in));
  p.counters = reinterpret_cast<unsigned int *>(split + (size_t)64 * (d_out + d_in) + (size_t)48 * d_in);
  p.ncounters = (d_out + kPM - 1) / kPM;
  return p;
}

void lr_u_planes(const void *cached, float *split, int d_out, int d_in, const uint16_t **u, const uint16_t **ut) {
  if (cached) {
    *u = static_cast<const uint16_t *>(cached);
    *ut = *u + (size_t)128 * d_in;
  } else {
    const LrPlanes pl = lr_planes(split, d_out, d_in);
    *u = pl.u;
    *ut = pl.ut;
  }
}

size_t lr_factor_planes_bytes(int d_in) { return (size_t)448 * d_in; }

cudaError_t launch_lr_factor_planes(const Launch &L, const float *U, int d_in, int rank, void *planes) {
  uint16_t *u = static_cast<uint16_t *>(planes);
  k_split_u<<<(d_in + 31) / 32, 256, 0, L.stream>>>(U, d_in, rank, 2, u, u + (size_t)128 * d_in, nullptr, 0);
  return cudaGetLastError();
}

bool lr_proj_tc_ok(const float *X, int d_in, const float *split) {
  return d_in % 32 == 0 && aligned16(X) && aligned16(split) && proj_encoder() != nullptr;
}

cudaError_t launch_lr_split_u_all(const Launch &L, const float *U, int d_out, int d_in, int rank, int nplanes_apply,
                                  float *split) {
  const LrPlanes pl = lr_planes(split, d_out, d_in);
  const int grid = (d_in + 31) / 32;
  k_split_u<<<grid, 256, 0, L.stream>>>(U, d_in, rank, nplanes_apply, pl.u, pl.ut, pl.counters, pl.ncounters);
  return cudaGetLastError();
}

cudaError_t launch_lr_proj_tc(const Launch &L, const float *X, int d_out, int d_in, const float *mu,
                              const float *sigma, int rank, bool inverse, bool tc_precision, float *part, float *Pc,
                              float *split, const uint16_t *ut_planes) {
  const LrPlanes pl = lr_planes(split, d_out, d_in);
  CUtensorMap tmX, tmUT;
  if (!map2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, X, (uint64_t)d_out, (uint64_t)d_in, 32, kPM) ||
      !map2d(&tmUT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ut_planes, 96, (uint64_t)d_in, kPK, 32))
    return cudaErrorInvalidValue;
  ProjParams P;
  P.mu = mu;
  P.sigma = sigma;
  P.rank = rank;
  P.d_out = d_out;
  P.d_in = d_in;
  P.inverse = inverse;
  P.nsplit = lr_proj_tc_splits(L.sms, d_out, d_in);
  P.ktiles = (d_in + kPK - 1) / kPK;
  P.part = part;
  P.Pc = Pc;
  P.pc_planes = pl.pc;
  P.pc_nplanes = tc_precision ? 1 : 2;
  P.counters = pl.counters;
  const int grid = pl.ncounters * P.nsplit;
  cudaError_t e;
  const int smem = (tc_precision ? PLayout<2>::total : PLayout<3>::total) + 1024;
  auto kern = tc_precision ? k_lr_proj_tc<2> : k_lr_proj_tc<3>;
  if (tc_precision) e = ensure_dynamic_smem<k_lr_proj_tc<2>>(smem);
  else e = ensure_dynamic_smem<k_lr_proj_tc<3>>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (P.nsplit > 1) ? 1 : 0;   // the grid barrier needs every CTA resident
  return cudaLaunchKernelEx(&cfg, kern, P, tmX, tmUT, L.status);
}

}  // namespace gift
