// One-pass rank-r encode: W is read from HBM once.
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17): W~ = sigma^-1/2 W +
// ((W U) diag(c)) U^T, c = mu^-1/2 - sigma^-1/2, then the per-tensor amax scale and the FP8
// (or NVFP4) pack.  The two-kernel form streams W three times (projection, amax, pack) or
// twice (projection, fused encode); here each CTA keeps its part of W on chip from the
// projection to the pack.
//
// CTA = one 128-row block x at most 8 column tiles of 64 (the same slice of W the projection
// sums over).  Tiles 0-3 stay in shared memory (32 KB each), tiles 4-7 in tensor memory
// (64 columns each).  Cooperative launch (all CTAs resident) with three clock-bounded
// grid-wide barriers:
//   phase 1  TMA W tile + U^T term planes; warps 0-7 split the tile exactly into BF16 terms
//            (TMEM A operand, double-buffered) and, for tiles 4-7, store alpha W into the
//            tile's TMEM home; warp 9 runs the projection MMAs into a fresh accumulator per
//            tile, folded with round-to-nearest FP32 adds; the slice partial of P -> global.
//   barrier  every slice written.  Each CTA sums its share of its row block's rows over the
//            slices (slice order, compensated FP32, c in FP64) -> Pc and its term planes.
//   barrier  Pc complete.  phase 2: TMA the Pc planes (A, shared memory) and the U planes of
//            each tile (B); MMA D = Pc U^T: tiles 0-3 into fresh accumulators (then
//            W~ = fma(alpha, W, D) from the shared-memory copy of W), tiles 4-7 accumulated
//            onto alpha W in their homes; CTA amax.
//   barrier  tensor amax (skipped with a caller amax).  phase 3: pack out of tensor memory.
// The projection arithmetic (terms, products, per-tile folding, slice sums) is the same as
// the tensor-core projection kernel's, so Pc is the same; tiles 0-3 use the same W~
// arithmetic as the two-kernel path, tiles 4-7 add Pc U^T onto the rounded alpha W.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kOM = 128, kON = 64;
constexpr int kOMaxTiles = 8;
constexpr int kOSmemHomes = 4;
constexpr int kOWarps = 8;
constexpr int kOThreads = 32 * (kOWarps + 2);
constexpr int kOBox = 128 * 128;        // 128 rows x 32 FP32
constexpr int kOTile = 2 * kOBox;       // 32 KB
constexpr int kOUtBox = 32 * 128;       // U^T plane box: 32 rows x 64 BF16
constexpr int kOUBox = 64 * 128;        // U plane box: 64 rows x 128 bytes
constexpr int kOAPlane = 128 * 128;     // Pc plane box: 128 rows x 128 bytes
constexpr int kOffHome = 0;                                   // tiles 0-3
constexpr int kOffStage = kOffHome + kOSmemHomes * kOTile;    // phase 1: 2 staging tiles
constexpr int kOffPcA = kOffStage;                            // phase 2: Pc planes
constexpr int kOffURing = kOffStage + 2 * kOAPlane;           // phase 2: 3 x U planes
constexpr int kOUSlots = 3;
constexpr int kOffUtRing = kOffStage + 2 * kOTile;            // phase 1: 2 x U^T planes
constexpr int kOSmemTotal = kOffUtRing + 2 * 3 * kOUtBox;     // 216 KB
constexpr uint32_t kOTmHome = 0;     // tiles 4-7
constexpr uint32_t kOTmABuf = 256;   // phase 1: A buffers (2 x 96 columns)
constexpr uint32_t kOTmPAcc = 448;   // phase 1: P accumulators (2 x 32 columns)
constexpr uint32_t kOTmD = 256;      // phase 2/3: W~ of tiles 0-3 (4 x 64 columns)
constexpr long long kOWait = 4000000000LL;

struct OnePassParams {
  LrApply a;
  const float *mu;
  int tiles_n, cpr;
  float *part;                 // cpr x d_out x 32 slice partials
  float *Pc;                   // d_out x 32
  uint16_t *pc_planes;         // term planes of Pc (NT - 1 planes)
  unsigned int *grid_counter;  // zero on entry
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}
__device__ __forceinline__ int sw(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }
// phase-3 code staging (in the freed W homes): FP8 rows of 32 x 16 bytes, NVFP4 rows of
// 16 x 16 bytes, 16-byte chunks XOR-swizzled by row; NVFP4 block scales 32 bytes per row after
constexpr int kOStgScales = 128 * 256;
__device__ __forceinline__ int stg8(int r, int c) { return r * 512 + ((c ^ (r & 31)) << 4); }
__device__ __forceinline__ int stg4(int r, int c) { return r * 256 + ((c ^ (r & 15)) << 4); }

// Grid-wide barrier on a monotonic counter (one thread per CTA); false on timeout.
__device__ __forceinline__ bool grid_barrier(unsigned int *counter, unsigned int target) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
  const long long t0 = clock64();
  while (ld_acquire_u32(counter) < target)
    if (clock64() - t0 > kOWait) return false;
  return true;
}

}  // namespace

template <int EPI, int F, int NT, bool TOUT>
__global__ void __launch_bounds__(kOThreads, 1) k_lr_encode_onepass(const __grid_constant__ OnePassParams P,
                                                                    const __grid_constant__ CUtensorMap tmW,
                                                                    const __grid_constant__ CUtensorMap tmUT,
                                                                    const __grid_constant__ CUtensorMap tmU,
                                                                    const __grid_constant__ CUtensorMap tmPc,
                                                                    int *status) {
  constexpr int NPL = NT - 1;                        // Pc / U planes of the apply
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t wfull[kOMaxTiles], utfull[2], utempty[2], stgempty[2], afull[2], aempty[2], cfull[2], cempty[2];
  __shared__ uint64_t go2, pcfull, ufull[kOUSlots], uempty[kOUSlots], dfull[kOMaxTiles];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[kOWarps];
  __shared__ double coef[32];
  __shared__ float amax_sh;
  __shared__ volatile int failed;

  const LrApply &a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = a.d_out, d_in = a.d_in;
  const int rb = blockIdx.x / P.cpr, jc = blockIdx.x - rb * P.cpr;
  const int cb0 = (int)(((long long)P.tiles_n * jc) / P.cpr);
  const int nt = (int)(((long long)P.tiles_n * (jc + 1)) / P.cpr) - cb0;   // 1..8
  const int r0 = rb * kOM;
  const unsigned int G = gridDim.x;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < kOMaxTiles; ++i) {
      tc::mbar_init(&wfull[i], 1);
      tc::mbar_init(&dfull[i], 1);
    }
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&utfull[k], 1);
      tc::mbar_init(&utempty[k], 1);
      tc::mbar_init(&stgempty[k], kOWarps);
      tc::mbar_init(&afull[k], kOWarps);
      tc::mbar_init(&aempty[k], 1);
      tc::mbar_init(&cfull[k], 1);
      tc::mbar_init(&cempty[k], kOWarps);
    }
    for (int k = 0; k < kOUSlots; ++k) {
      tc::mbar_init(&ufull[k], 1);
      tc::mbar_init(&uempty[k], 1);
    }
    tc::mbar_init(&go2, 1);
    tc::mbar_init(&pcfull, 1);
    tc::fence_mbar_init();
    failed = 0;
  }
  if (warp == 1) {   // FP64 coefficients of the finalize
    const int k = lane;
    double c = 0.0;
    if (k < a.rank) {
      const double m = (double)P.mu[k], sg = (double)a.sigma[0];
      if (!(m > 0.0) || !(sg > 0.0)) {
        if (blockIdx.x == 0) set_status(status, GIFT_ERR_NOT_PD);
      } else {
        c = 1.0 / sqrt(m) - 1.0 / sqrt(sg);
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
    if (!tc::mbar_wait_bounded(bar, parity, kOWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kOWarps) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      auto load_w = [&](int i, uint8_t *dst) {
        const int c0 = (cb0 + i) * kON;
        tc::mbar_arrive_expect_tx(&wfull[i], kOTile);
        tc::tma_load_2d(dst, &tmW, c0, r0, &wfull[i]);
        tc::tma_load_2d(dst + kOBox, &tmW, c0 + 32, r0, &wfull[i]);
      };
      auto w_dst = [&](int i) {
        return i < kOSmemHomes ? sm + kOffHome + i * kOTile : sm + kOffStage + (i & 1) * kOTile;
      };
      // phase 1: every W tile with a free destination at once (homes, first use of each
      // staging buffer); the U^T planes through their two-slot ring; the second use of a
      // staging buffer once the splitters are done with its first tile
      const int first = nt < kOSmemHomes + 2 ? nt : kOSmemHomes + 2;
      for (int i = 0; i < first; ++i) load_w(i, w_dst(i));
      bool ok = true;
      for (int i = 0; i < nt && ok; ++i) {
        const int u = i & 1;
        if (!(ok = wait(&utempty[u], (uint32_t)(((i >> 1) & 1) ^ 1)))) break;
        tc::mbar_arrive_expect_tx(&utfull[u], NT * kOUtBox);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          tc::tma_load_2d(sm + kOffUtRing + u * 3 * kOUtBox + t * kOUtBox, &tmUT, (cb0 + i) * kON, 32 * t, &utfull[u]);
        const int i2 = i + 2;   // staging second use (tiles 6, 7) once tile i2 - 2 has been split
        if (i >= kOSmemHomes && i2 < nt) {
          if (!(ok = wait(&stgempty[i2 & 1], 0))) break;
          load_w(i2, w_dst(i2));
        }
      }
      // phase 2: U planes of the first tiles into the freed region as soon as phase 1 is done
      // with it (the last U^T reads and the last staging reads), Pc once the grid has written it
      if (ok) {
        for (int u = 0; u < 2 && u < nt; ++u) ok = ok && wait(&utempty[u], (uint32_t)((((nt - 1 - u) >> 1)) & 1));
        for (int k = 0; k < 2; ++k) {
          const int uses = (nt > kOSmemHomes + k) ? (nt - kOSmemHomes - k + 1) / 2 : 0;
          if (uses > 0) ok = ok && wait(&stgempty[k], (uint32_t)((uses - 1) & 1));
        }
      }
      auto load_u = [&](int i) {
        const int k = i % kOUSlots, c0 = (cb0 + i) * kON;
        tc::mbar_arrive_expect_tx(&ufull[k], NPL * kOUBox);
#pragma unroll
        for (int q = 0; q < NPL; ++q)
          tc::tma_load_2d(sm + kOffURing + k * 2 * kOUBox + q * kOUBox, &tmU, 0, q * d_in + c0, &ufull[k]);
      };
      if (ok) {
        for (int i = 0; i < nt && i < kOUSlots; ++i) load_u(i);
        if (wait(&go2, 0)) {
          fence_proxy_async_global();
          tc::mbar_arrive_expect_tx(&pcfull, NPL * kOAPlane);
#pragma unroll
          for (int q = 0; q < NPL; ++q)
            tc::tma_load_2d(sm + kOffPcA + q * kOAPlane, &tmPc, 0, q * d_out + r0, &pcfull);
          for (int i = kOUSlots; i < nt; ++i) {
            if (!wait(&uempty[i % kOUSlots], (uint32_t)(((i / kOUSlots) - 1) & 1))) break;
            load_u(i);
          }
        }
      }
    }
  } else if (warp == kOWarps + 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      // phase 1: P tile = X terms (TMEM) x U^T terms (shared memory), K = 64
      {
        constexpr uint32_t idesc = tc::idesc_bf16(kOM, 32);
        constexpr int np = (NT == 2) ? 3 : 6;
        constexpr int pa[6] = {NT == 2 ? 1 : 2, NT == 2 ? 0 : 1, 0, 1, 0, 0};
        constexpr int pb[6] = {0, 1, NT == 2 ? 0 : 2, 0, 1, 0};
        for (int i = 0; i < nt; ++i) {
          const int b = i & 1;
          if (!wait(&utfull[b], (uint32_t)((i >> 1) & 1))) break;
          if (!wait(&afull[b], (uint32_t)((i >> 1) & 1))) break;
          if (!wait(&cempty[b], (uint32_t)(((i >> 1) & 1) ^ 1))) break;
          tc::fence_after_sync();
          const uint32_t ub = tc::smem_u32(sm + kOffUtRing + b * 3 * kOUtBox);
          uint32_t acc = 0;
#pragma unroll
          for (int p = 0; p < np; ++p) {
#pragma unroll
            for (int k = 0; k < kON / 16; ++k) {
              tc::mma_bf16_ta(tmem + kOTmPAcc + 32 * b, tmem + kOTmABuf + 96 * b + 32 * pa[p] + 8 * k,
                              tc::sdesc_kmajor_sw128(ub + pb[p] * kOUtBox + 32 * k), idesc, acc);
              acc = 1;
            }
          }
          tc::mma_commit(&utempty[b]);
          tc::mma_commit(&aempty[b]);
          tc::mma_commit(&cfull[b]);
        }
      }
      // phase 2: D = Pc U^T (A = Pc planes, B = U planes), K = 32
      if (wait(&pcfull, 0)) {
        tc::fence_after_sync();
        constexpr uint32_t idesc = tc::idesc_bf16(kOM, kON);
        constexpr int np = (NPL == 1) ? 3 : 6;
        constexpr int pa[6] = {NPL == 1 ? 1 : 2, NPL == 1 ? 0 : 1, 0, 1, 0, 0};
        constexpr int pb[6] = {0, 1, NPL == 1 ? 0 : 2, 0, 1, 0};
        const uint32_t a0 = tc::smem_u32(sm + kOffPcA);
        for (int i = 0; i < nt; ++i) {
          const int u = i % kOUSlots;
          if (!wait(&ufull[u], (uint32_t)((i / kOUSlots) & 1))) break;
          tc::fence_after_sync();
          const uint32_t b0 = tc::smem_u32(sm + kOffURing + u * 2 * kOUBox);
          const bool home_tmem = i >= kOSmemHomes;
          const uint32_t d = home_tmem ? tmem + kOTmHome + (uint32_t)(64 * (i - kOSmemHomes))
                                       : tmem + kOTmD + (uint32_t)(64 * i);
          uint32_t acc = home_tmem ? 1u : 0u;   // tiles 4-7: add onto alpha W
#pragma unroll
          for (int p = 0; p < np; ++p) {
            const uint32_t aa = a0 + (pa[p] >> 1) * kOAPlane + 64 * (pa[p] & 1);
            const uint32_t bb = b0 + (pb[p] >> 1) * kOUBox + 64 * (pb[p] & 1);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              tc::mma_bf16(d, tc::sdesc_kmajor_sw128(aa + 32 * k), tc::sdesc_kmajor_sw128(bb + 32 * k), idesc, acc);
              acc = 1;
            }
          }
          tc::mma_commit(&uempty[u]);
          tc::mma_commit(&dfull[i]);
        }
      }
    }
  } else {
    // ======================= workers (warps 0-7): thread = row, 32 columns =======================
    const int quarter = warp & 3, half = warp >> 2;
    const int lr = quarter * 32 + lane, row = r0 + lr;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float alpha = (float)(1.0 / sqrt((double)a.sigma[0]));

    // ---------------- phase 1: projection ----------------
    float accp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) accp[j] = 0.0f;
    auto fold = [&](int j) {
      const int c = j & 1;
      wait(&cfull[c], (uint32_t)((j >> 1) & 1));
      tc::fence_after_sync();
      uint32_t raw[16];
      tc::tmem_ld16_nowait(tmem + lane_off + kOTmPAcc + 32 * c + 16 * half, raw);
      tc::tmem_wait_ld16(raw);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&cempty[c]);
#pragma unroll
      for (int q = 0; q < 16; ++q) accp[q] = __fadd_rn(accp[q], __uint_as_float(raw[q]));
    };
    for (int i = 0; i < nt; ++i) {
      const int b = i & 1;
      wait(&wfull[i], 0);
      wait(&aempty[b], (uint32_t)(((i >> 1) & 1) ^ 1));
      tc::fence_after_sync();
      const uint8_t *box = (i < kOSmemHomes ? sm + kOffHome + i * kOTile : sm + kOffStage + (i & 1) * kOTile) +
                           half * kOBox;
      float x[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 v = *reinterpret_cast<const float4 *>(box + sw(lr, c));
        x[4 * c] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
      }
      uint32_t w1[16], w2[16], w3[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        uint16_t a1, a2, a3, b1, b2, b3;
        tc::bf16_split3(x[2 * q], a1, a2, a3);
        tc::bf16_split3(x[2 * q + 1], b1, b2, b3);
        w1[q] = (uint32_t)a1 | ((uint32_t)b1 << 16);
        w2[q] = (uint32_t)a2 | ((uint32_t)b2 << 16);
        w3[q] = (uint32_t)a3 | ((uint32_t)b3 << 16);
      }
      const uint32_t abase = tmem + lane_off + kOTmABuf + 96 * b + 16 * half;
      tc::tmem_st16(abase, w1);
      tc::tmem_st16(abase + 32, w2);
      if (NT == 3) tc::tmem_st16(abase + 64, w3);
      if (i >= kOSmemHomes) {
        uint32_t aw[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) aw[q] = __float_as_uint(__fmul_rn(alpha, x[q]));
        const uint32_t home = tmem + lane_off + kOTmHome + (uint32_t)(64 * (i - kOSmemHomes) + 32 * half);
        tc::tmem_st16(home, aw);
        tc::tmem_st16(home + 16, aw + 16);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();   // staging is refilled by TMA
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&afull[b]);
        if (i >= kOSmemHomes) tc::mbar_arrive(&stgempty[i & 1]);
      }
      if (i > 0) fold(i - 1);
    }
    fold(nt - 1);
    if (row < d_out) {
      float4 *dst = reinterpret_cast<float4 *>(P.part + ((size_t)jc * d_out + row) * 32 + 16 * half);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(accp[4 * q], accp[4 * q + 1], accp[4 * q + 2], accp[4 * q + 3]);
    }
    __threadfence();
    tc::named_bar_sync(1, 32 * kOWarps);
    if (tid == 0 && !grid_barrier(P.grid_counter, G)) set_status(status, GIFT_ERR_TIMEOUT);
    tc::named_bar_sync(1, 32 * kOWarps);

    // ---------------- this CTA's share of Pc (rows of its row block) ----------------
    {
      const int ra = r0 + (kOM * jc) / P.cpr, rz = r0 + (kOM * (jc + 1)) / P.cpr;
      for (int item = tid; item < (rz - ra) * 8; item += 32 * kOWarps) {
        const int rr = ra + (item >> 3), kb = 4 * (item & 7);
        if (rr >= d_out) continue;
        float sum[4] = {0.f, 0.f, 0.f, 0.f}, comp[4] = {0.f, 0.f, 0.f, 0.f};
        for (int q0 = 0; q0 < P.cpr; q0 += 16) {
          float4 xs4[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (q0 + u < P.cpr)
              xs4[u] = __ldcg(reinterpret_cast<const float4 *>(P.part + ((size_t)(q0 + u) * d_out + rr) * 32 + kb));
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (q0 + u < P.cpr) {
              const float xs[4] = {xs4[u].x, xs4[u].y, xs4[u].z, xs4[u].w};
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
#pragma unroll
        for (int e = 0; e < 4; ++e) tc::write_term_planes(P.pc_planes, (size_t)d_out, (size_t)rr, kb + e, pc[e], NPL);
      }
    }
    fence_proxy_async_global();   // the planes are read back by TMA
    __threadfence();
    tc::named_bar_sync(1, 32 * kOWarps);
    if (tid == 0) {
      if (!grid_barrier(P.grid_counter, 2 * G)) set_status(status, GIFT_ERR_TIMEOUT);
      tc::mbar_arrive(&go2);
    }

    // ---------------- phase 2: W~ of every tile, CTA amax ----------------
    // software-pipelined: the next tile's TMEM load is issued before this tile's store-back
    // (tcgen05.wait::ld waits for all of a thread's loads, so it is issued once per tile);
    // the stores are waited for once, before phase 3 reads the slots again
    uint32_t m_run = 0;
    auto d_slot = [&](int i) {
      return tmem + lane_off + ((i < kOSmemHomes) ? kOTmD + (uint32_t)(64 * i) : kOTmHome + (uint32_t)(64 * (i - kOSmemHomes))) +
             (uint32_t)(32 * half);
    };
    uint32_t nxt[32];
    wait(&dfull[0], 0);
    tc::fence_after_sync();
    tc::tmem_ld32_nowait(d_slot(0), nxt);
    for (int i = 0; i < nt; ++i) {
      const int c0 = (cb0 + i) * kON;
      float4 w[8];
      if (i < kOSmemHomes) {
        const uint8_t *box = sm + kOffHome + i * kOTile + half * kOBox;
#pragma unroll
        for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const float4 *>(box + sw(lr, c));
      }
      tc::tmem_wait_ld(nxt);
      uint32_t raw[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) raw[e] = nxt[e];
      if (i + 1 < nt) {
        wait(&dfull[i + 1], 0);
        tc::fence_after_sync();
        tc::tmem_ld32_nowait(d_slot(i + 1), nxt);
      }
      if (i < kOSmemHomes) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          raw[4 * c + 0] = __float_as_uint(fmaf(alpha, w[c].x, __uint_as_float(raw[4 * c + 0])));
          raw[4 * c + 1] = __float_as_uint(fmaf(alpha, w[c].y, __uint_as_float(raw[4 * c + 1])));
          raw[4 * c + 2] = __float_as_uint(fmaf(alpha, w[c].z, __uint_as_float(raw[4 * c + 2])));
          raw[4 * c + 3] = __float_as_uint(fmaf(alpha, w[c].w, __uint_as_float(raw[4 * c + 3])));
        }
        tc::tmem_st16(d_slot(i), raw);
        tc::tmem_st16(d_slot(i) + 16, raw + 16);
      }
      if (row < d_out && (c0 + 32 * half) < d_in) {
#pragma unroll
        for (int e = 0; e < 32; ++e) m_run = max(m_run, raw[e] & 0x7FFFFFFFu);
        if (TOUT) {
          float4 *dst = reinterpret_cast<float4 *>(a.tout + (size_t)row * d_in + c0 + 32 * half);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            dst[c] = make_float4(__uint_as_float(raw[4 * c]), __uint_as_float(raw[4 * c + 1]),
                                 __uint_as_float(raw[4 * c + 2]), __uint_as_float(raw[4 * c + 3]));
        }
      }
    }
    tc::tmem_wait_st();
    m_run = warp_max_u32(m_run);
    if (lane == 0) red[warp] = m_run;
    tc::named_bar_sync(1, 32 * kOWarps);
    if (tid == 0) {
      uint32_t m = 0;
      for (int w = 0; w < kOWarps; ++w) m = max(m, red[w]);
      float amax;
      if (a.amax_in) {
        amax = a.amax_in[0];
      } else {
        if (m) atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws), m);
        if (!grid_barrier(P.grid_counter, 3 * G)) set_status(status, GIFT_ERR_TIMEOUT);
        amax = __uint_as_float(ld_acquire_u32(reinterpret_cast<const unsigned int *>(a.amax_ws)));
      }
      amax_sh = amax;
      if (blockIdx.x == 0) {
        if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
        if (EPI == LR_PACK_TENSOR) reinterpret_cast<float *>(a.scales)[0] = scale_pair(amax, fmax_of<F>()).s;
        else a.tscale[0] = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
        if (a.amax_out) a.amax_out[0] = amax;
      }
    }
    tc::named_bar_sync(1, 32 * kOWarps);
    const float amax = amax_sh;
    const ScalePair sp = scale_pair(amax, fmax_of<F>());
    const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);

    // ---------------- phase 3: pack out of tensor memory (next tile's load in flight) ----------------
    auto slot_of = [&](int i) {
      return tmem + lane_off + ((i < kOSmemHomes) ? kOTmD + (uint32_t)(64 * i) : kOTmHome + (uint32_t)(64 * (i - kOSmemHomes))) +
             (uint32_t)(32 * half);
    };
    tc::tmem_ld32_nowait(slot_of(0), nxt);
    for (int i = 0; i < nt; ++i) {
      const int c0 = (cb0 + i) * kON;
      tc::tmem_wait_ld(nxt);
      uint32_t raw[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) raw[e] = nxt[e];
      if (i + 1 < nt) tc::tmem_ld32_nowait(slot_of(i + 1), nxt);
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
      // codes are staged in shared memory (the W homes are free now) for coalesced row stores
      if (EPI == LR_PACK_TENSOR) {
        uint32_t w4[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float *x = v + 4 * h;
          w4[h] = pack4_fp8<F>(__fmul_rn(x[0], sp.m), __fmul_rn(x[1], sp.m), __fmul_rn(x[2], sp.m),
                               __fmul_rn(x[3], sp.m));
        }
        const int c = 4 * i + 2 * half;   // 16-byte chunk of the CTA's 512-byte code row
        *reinterpret_cast<uint4 *>(sm + stg8(lr, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        *reinterpret_cast<uint4 *>(sm + stg8(lr, c + 1)) = make_uint4(w4[4], w4[5], w4[6], w4[7]);
      } else {
        uint16_t sc = 0;
        uint32_t cw[4];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t gm = 0;
#pragma unroll
          for (int e = 0; e < 16; ++e) gm = max(gm, abs_bits(v[16 * g + e]));
          const Nv4Group grp = nvfp4_group(__uint_as_float(gm), s_t);
          float y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] = __fmul_rn(v[16 * g + e], grp.r);
          cw[2 * g] = pack8_e2m1(y);
          cw[2 * g + 1] = pack8_e2m1(y + 8);
          sc |= (uint16_t)grp.e_code << (8 * g);
        }
        *reinterpret_cast<uint4 *>(sm + stg4(lr, 2 * i + half)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        *reinterpret_cast<uint16_t *>(sm + kOStgScales + lr * 32 + 4 * i + 2 * half) = sc;
      }
    }
    // coalesced copy-out of the CTA's code rows (and NVFP4 block scales)
    tc::named_bar_sync(1, 32 * kOWarps);
    const int cbase = cb0 * kON;
    if (EPI == LR_PACK_TENSOR) {
      for (int r = warp; r < kOM; r += kOWarps) {
        const int gr = r0 + r, col = cbase + 16 * lane;
        if (gr < d_out && lane < 4 * nt && col < d_in)
          *reinterpret_cast<uint4 *>(a.codes + (size_t)gr * d_in + col) = *reinterpret_cast<const uint4 *>(sm + stg8(r, lane));
      }
    } else {
      for (int item = tid; item < kOM * 16; item += 32 * kOWarps) {
        const int r = item >> 4, c = item & 15, gr = r0 + r, col = cbase + 32 * c;
        if (gr < d_out && c < 2 * nt && col < d_in)
          *reinterpret_cast<uint4 *>(a.codes + (((size_t)gr * d_in + col) >> 1)) = *reinterpret_cast<const uint4 *>(sm + stg4(r, c));
      }
      for (int item = tid; item < kOM * 16; item += 32 * kOWarps) {
        const int r = item >> 4, q = item & 15, gr = r0 + r, col = cbase + 32 * q;   // two scale bytes per 32 columns
        if (gr < d_out && q < 2 * nt && col < d_in)
          *reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(a.scales) + (size_t)gr * (d_in / kNvGroup) + col / kNvGroup) =
              *reinterpret_cast<const uint16_t *>(sm + kOStgScales + r * 32 + 2 * q);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 onepass_encoder() {
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

bool omap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t rows, uint64_t cols,
          uint32_t box_cols, uint32_t box_rows) {
  auto enc = onepass_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs per row block: at most kOMaxTiles tiles each, the CTA's column range being its slice.
int onepass_plan(int sms, int d_out, int d_in, int *cpr_out) {
  const int tiles_n = (d_in + kON - 1) / kON;
  const int tiles_m = (d_out + kOM - 1) / kOM;
  if (tiles_m > sms) return 0;
  int cpr = (tiles_n + kOMaxTiles - 1) / kOMaxTiles;
  const int spread = sms / tiles_m;
  if (spread > cpr) cpr = spread < tiles_n ? spread : tiles_n;
  if ((long long)cpr * tiles_m > sms) return 0;
  *cpr_out = cpr;
  return cpr * tiles_m;
}

template <int EPI, int F, int NT, bool TOUT>
cudaError_t onepass_launch(const Launch &L, const OnePassParams &P, int grid) {
  const LrApply &a = P.a;
  const LrPlanes pl = lr_planes(a.split, a.d_out, a.d_in);
  constexpr int NPL = NT - 1;
  CUtensorMap tmW, tmUT, tmU, tmPc;
  if (!omap(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.X, (uint64_t)a.d_out, (uint64_t)a.d_in, 32, kOM) ||
      !omap(&tmUT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.ut_planes, 96, (uint64_t)a.d_in, kON, 32) ||
      !omap(&tmU, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.u_planes, (uint64_t)NPL * a.d_in, 32, 32, kON) ||
      !omap(&tmPc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pl.pc, (uint64_t)NPL * a.d_out, 32, 32, kOM))
    return cudaErrorInvalidValue;
  const int smem = kOSmemTotal + 1024;
  auto kern = k_lr_encode_onepass<EPI, F, NT, TOUT>;
  cudaError_t e;
  if ((e = ensure_dynamic_smem<k_lr_encode_onepass<EPI, F, NT, TOUT>>(smem)) != cudaSuccess) return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kOThreads, smem)) != cudaSuccess) return e;
  if (per_sm < 1 || grid > per_sm * L.sms) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kOThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P, tmW, tmUT, tmU, tmPc, L.status);
}

template <int NT>
cudaError_t onepass_dispatch(const Launch &L, int epi, int fmt, const OnePassParams &P, int grid) {
  const bool t = P.a.tout != nullptr;
  if (epi == LR_NVFP4)
    return t ? onepass_launch<LR_NVFP4, FMT_E4M3, NT, true>(L, P, grid)
             : onepass_launch<LR_NVFP4, FMT_E4M3, NT, false>(L, P, grid);
  if (fmt == GIFT_FMT_E5M2)
    return t ? onepass_launch<LR_PACK_TENSOR, FMT_E5M2, NT, true>(L, P, grid)
             : onepass_launch<LR_PACK_TENSOR, FMT_E5M2, NT, false>(L, P, grid);
  return t ? onepass_launch<LR_PACK_TENSOR, FMT_E4M3, NT, true>(L, P, grid)
           : onepass_launch<LR_PACK_TENSOR, FMT_E4M3, NT, false>(L, P, grid);
}

}  // namespace

bool lr_encode_onepass_ok(const Launch &L, const LrApply &a, int epi, const float *part, size_t part_floats) {
  if (epi != LR_PACK_TENSOR && epi != LR_NVFP4) return false;
  if (a.inverse || !a.split || !a.grid_counter || !part) return false;
  if (!lr_apply_tc_ok(a, epi) || !lr_proj_tc_ok(a.X, a.d_in, a.split) || onepass_encoder() == nullptr) return false;
  int cpr = 0;
  if (onepass_plan(L.sms, a.d_out, a.d_in, &cpr) <= 0) return false;
  return (size_t)cpr * a.d_out * 32 <= part_floats;
}

// U planes (and the zeroed counters) must be in a.split, a.amax_ws zero without a caller
// amax, a.grid_counter zero.
cudaError_t launch_lr_encode_onepass(const Launch &L, int epi, int fmt, const LrApply &a, const float *mu,
                                     float *part, float *Pc) {
  int cpr = 0;
  const int grid = onepass_plan(L.sms, a.d_out, a.d_in, &cpr);
  if (grid <= 0) return cudaErrorInvalidValue;
  OnePassParams P;
  P.a = a;
  P.mu = mu;
  P.tiles_n = (a.d_in + kON - 1) / kON;
  P.cpr = cpr;
  P.part = part;
  P.Pc = Pc;
  P.pc_planes = lr_planes(a.split, a.d_out, a.d_in).pc;
  P.grid_counter = a.grid_counter;
  return a.terms == 1 ? onepass_dispatch<2>(L, epi, fmt, P, grid) : onepass_dispatch<3>(L, epi, fmt, P, grid);
}

}  // namespace gift
