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
// (64 columns each).  Cooperative launch (all CTAs resident) with clock-bounded grid-wide
// barriers on one monotonic counter.  Per tensor:
//   phase 1  TMA W tile + U^T term planes; warps 0-7 split the tile exactly into BF16 terms
//            (TMEM A operand, double-buffered) and, for tiles 4-7, store alpha W into the
//            tile's TMEM home; warp 9 runs the projection MMAs into a fresh accumulator per
//            tile, folded with round-to-nearest FP32 adds; the slice partial of P -> global.
//   barrier  every slice written.  Each CTA sums its share of its row block's rows over the
//            slices (slice order, compensated FP32, c in FP64) -> Pc and its term planes.
//   barrier  Pc complete.  The workers put alpha W of tiles 0-3 into tensor memory (columns
//            256-511, free after phase 1) while the Pc planes (A, shared memory) arrive.
//            phase 2: two groups of four tiles, each one N = 256 MMA chain with the group's
//            U planes as B (one 256-row box per plane): W~ = alpha W + Pc U^T accumulated in
//            tensor memory, tiles 0-3 in columns 256-511, tiles 4-7 in their homes; CTA amax.
//   barrier  tensor amax (skipped with a caller amax).  phase 3: pack out of tensor memory,
//            codes staged in shared memory for coalesced row stores.
// One launch encodes a batch of tensors that share the factor (the data-parallel replicas of
// a layer's gradient): the rings and barriers run on across the batch, and the next tensor's
// tiles 0-3 are fetched into their shared-memory homes while this tensor is still in phase
// 2, its amax barrier and its pack (the homes are free once alpha W has moved to tensor
// memory; the codes are staged in the phase-2 region).
// The projection arithmetic (terms, products, per-tile folding, slice sums) is the same as
// the tensor-core projection kernel's, so Pc is the same; W~ is Pc U^T added by the tensor
// cores onto the rounded alpha W (the two-kernel path rounds one fma instead).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

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
constexpr int kOGroupTiles = 4;          // phase 2: tiles per MMA group (N = 256)
constexpr int kOUGroup = kOGroupTiles * kON * 128;   // U plane box of a group: 256 rows x 128 bytes
static_assert(kOGroupTiles == kOSmemHomes, "phase-2 groups: the shared-memory tiles, then the tensor-memory tiles");
constexpr int kOAPlane = 128 * 128;     // Pc plane box: 128 rows x 128 bytes
constexpr int kOffHome = 0;                                   // tiles 0-3
constexpr int kOffStage = kOffHome + kOSmemHomes * kOTile;    // phase 1: 2 staging tiles
constexpr int kOffPcA = kOffStage;                            // phase 2: Pc planes
constexpr int kOffURing = kOffStage + 2 * kOAPlane;           // phase 2: U planes of a group
constexpr int kOffUtRing = kOffStage + 2 * kOTile;            // phase 1: 2 x U^T planes
constexpr int kOSmemTotal = kOffURing + 2 * kOUGroup;         // 224 KB
static_assert(kOffUtRing + 2 * 3 * kOUtBox <= kOSmemTotal, "U^T ring outside the allocation");
constexpr uint32_t kOTmHome = 0;     // tiles 4-7
constexpr uint32_t kOTmABuf = 256;   // phase 1: A buffers (2 x 96 columns)
constexpr uint32_t kOTmPAcc = 448;   // phase 1: P accumulators (2 x 32 columns)
constexpr uint32_t kOTmD = 256;      // phase 2/3: W~ of tiles 0-3 (4 x 64 columns)
constexpr long long kOWait = 4000000000LL;

struct OnePassParams {
  LrApply a;                   // shared: factor, planes, shapes; a.amax_ws = one word per tensor
  const float *mu;
  int tiles_n, cpr, nb;        // nb tensors in the batch
  float *part;                 // cpr x d_out x 32 slice partials
  float *Pc;                   // d_out x 32
  uint16_t *pc_planes;         // term planes of Pc (NT - 1 planes)
  unsigned int *grid_counter;  // zero on entry
  LrEncodeItem item[kOnePassMaxBatch];
};
struct OnePassMaps {
  CUtensorMap w[kOnePassMaxBatch];   // W of each tensor
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
// phase-3 code staging (in the phase-2 region): FP8 rows of 32 x 16 bytes, NVFP4 rows of
// 16 x 16 bytes, 16-byte chunks XOR-swizzled by row; NVFP4 block scales 32 bytes per row after
constexpr int kOffCodes = kOffStage;
constexpr int kOStgScales = 128 * 256;
static_assert(kOffCodes + 128 * 512 <= kOffUtRing, "code staging overlaps the U^T ring");
__device__ __forceinline__ int stg8(int r, int c) { return r * 512 + ((c ^ (r & 31)) << 4); }
__device__ __forceinline__ int stg4(int r, int c) { return r * 256 + ((c ^ (r & 15)) << 4); }

}  // namespace

template <int EPI, int F, int NT, bool TOUT>
__global__ void __launch_bounds__(kOThreads, 1) k_lr_encode_onepass(const __grid_constant__ OnePassParams P,
                                                                    const __grid_constant__ OnePassMaps M,
                                                                    const __grid_constant__ CUtensorMap tmUT,
                                                                    const __grid_constant__ CUtensorMap tmU,
                                                                    const __grid_constant__ CUtensorMap tmPc,
                                                                    int *status) {
  constexpr int NPL = NT - 1;                        // Pc / U planes of the apply
  constexpr int kStg = kOMaxTiles - kOSmemHomes;     // tiles that pass through the staging buffers
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  // per-tile barriers complete once per tensor (parity = tensor & 1); the rings (U^T planes,
  // A buffers, P accumulators, U planes) count tiles across the whole batch
  __shared__ uint64_t wfull[kOMaxTiles], dfull[2], sdone[kStg];
  // mdone[b]: the projection MMAs of the tile in slot b are complete, so its U^T slot and A
  // buffer are free and its accumulator is ready (one commit serves all three)
  __shared__ uint64_t utfull[2], mdone[2], afull[2], cempty[2];
  __shared__ uint64_t go2, pcfull, hfree, sfree, dinit, ufull[2];
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
  const int ngroups = nt > kOGroupTiles ? 2 : 1;   // phase-2 MMA groups
  // the two groups' U planes side by side when they fit (one plane each), else one region
  constexpr bool kGroupsApart = kOffURing + 2 * NPL * kOUGroup <= kOSmemTotal;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int i = 0; i < kOMaxTiles; ++i) tc::mbar_init(&wfull[i], 1);
    for (int i = 0; i < kStg; ++i) tc::mbar_init(&sdone[i], kOWarps);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&utfull[k], 1);
      tc::mbar_init(&mdone[k], 1);
      tc::mbar_init(&afull[k], kOWarps);
      tc::mbar_init(&cempty[k], kOWarps);
    }
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&ufull[k], 1);
      tc::mbar_init(&dfull[k], 1);
    }
    tc::mbar_init(&go2, 1);
    tc::mbar_init(&pcfull, 1);
    tc::mbar_init(&hfree, kOWarps);
    tc::mbar_init(&dinit, kOWarps);
    tc::mbar_init(&sfree, kOWarps);
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
      tc::prefetch_tensormap(&tmUT);
      tc::prefetch_tensormap(&tmU);
      tc::prefetch_tensormap(&tmPc);
      for (int k = 0; k < P.nb; ++k) tc::prefetch_tensormap(&M.w[k]);
      for (int k = 0; k < P.nb; ++k) {
        const CUtensorMap *mw = &M.w[k];
        const uint32_t kp = (uint32_t)(k & 1), pp = kp ^ 1u;   // this tensor's / the previous one's parity
        const int g0 = k * nt;                                 // ring index of this tensor's tile 0
        auto load_w = [&](int i, uint8_t *dst) {
          const int c0 = (cb0 + i) * kON;
          tc::mbar_arrive_expect_tx(&wfull[i], kOTile);
          tc::tma_load_2d(dst, mw, c0, r0, &wfull[i]);
          tc::tma_load_2d(dst + kOBox, mw, c0 + 32, r0, &wfull[i]);
        };
        auto load_ut = [&](int i) {
          const int g = g0 + i, u = g & 1;
          if (!wait(&mdone[u], (uint32_t)(((g >> 1) & 1) ^ 1))) return false;
          tc::mbar_arrive_expect_tx(&utfull[u], NT * kOUtBox);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            tc::tma_load_2d(sm + kOffUtRing + u * 3 * kOUtBox + t * kOUtBox, &tmUT, (cb0 + i) * kON, 32 * t, &utfull[u]);
          return true;
        };
        // phase 2 B operand: the U planes of a group of up to four tiles (one 256-row box
        // per plane; rows past the CTA's tiles are loaded but not used)
        auto load_group = [&](int grp, uint8_t *dst) {
          tc::mbar_arrive_expect_tx(&ufull[grp], NPL * kOUGroup);
#pragma unroll
          for (int q = 0; q < NPL; ++q)
            tc::tma_load_2d(dst + q * kOUGroup, &tmU, 0, q * d_in + (cb0 + kOGroupTiles * grp) * kON, &ufull[grp]);
        };
        // phase 1: the home tiles as soon as the previous tensor's phase 2 has read its homes;
        // the first U^T planes once its phase-2 MMAs are done (their ring overlaps the U
        // ring); the staging tiles once its codes have left the staging region; the second
        // use of a staging buffer once the splitters are done with its first tile
        if (k > 0 && !wait(&hfree, pp)) break;
        for (int i = 0; i < nt && i < kOSmemHomes; ++i) load_w(i, sm + kOffHome + i * kOTile);
        if (k > 0 && !wait(&dfull[ngroups - 1], pp)) break;
        bool ok = true;
        for (int i = 0; i < nt && i < 2 && ok; ++i) ok = load_ut(i);
        if (!ok || (k > 0 && !wait(&sfree, pp))) break;
        for (int i = kOSmemHomes; i < nt && i < kOSmemHomes + 2; ++i) load_w(i, sm + kOffStage + (i & 1) * kOTile);
        for (int i = 2; i < nt && ok; ++i) {
          if (!(ok = load_ut(i))) break;
          if (i >= kOSmemHomes && i + 2 < nt) {
            if (!(ok = wait(&sdone[i - kOSmemHomes], kp))) break;
            load_w(i + 2, sm + kOffStage + (i & 1) * kOTile);
          }
        }
        if (!ok) break;
        // phase 2: the first group's U planes into the phase-1 region once phase 1 is done with
        // it (the last U^T reads and the last staging reads); Pc once the grid has written it;
        // the second group beside the first where both fit (one plane each), else in its place
        // once the first group's MMAs are done
        for (int u = 0; u < 2 && u < nt && ok; ++u) {
          const int g = g0 + nt - 1 - u;
          ok = wait(&mdone[g & 1], (uint32_t)((g >> 1) & 1));
        }
        for (int i = kOSmemHomes; i < nt && ok; ++i) ok = wait(&sdone[i - kOSmemHomes], kp);
        if (!ok) break;
        load_group(0, sm + kOffURing);
        if (ngroups == 2 && kGroupsApart) load_group(1, sm + kOffURing + NPL * kOUGroup);
        if (!wait(&go2, kp)) break;
        fence_proxy_async_global();
        tc::mbar_arrive_expect_tx(&pcfull, NPL * kOAPlane);
#pragma unroll
        for (int q = 0; q < NPL; ++q) tc::tma_load_2d(sm + kOffPcA + q * kOAPlane, &tmPc, 0, q * d_out + r0, &pcfull);
        if (ngroups == 2 && !kGroupsApart) {
          if (!wait(&dfull[0], kp)) break;   // the first group's MMAs are done with the region
          load_group(1, sm + kOffURing);
        }
      }
    }
  } else if (warp == kOWarps + 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      // shared-memory descriptors of the ring slots, formed once: each MMA adds a constant
      // (the start-address field counts 16-byte units), which keeps the issue loop short
      const uint64_t ut_desc0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kOffUtRing));
      const uint64_t pc_desc = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kOffPcA));
      const uint64_t u_desc0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kOffURing));
      for (int k = 0; k < P.nb && !failed; ++k) {
        const int g0 = k * nt;
        // phase 1: P tile = X terms (TMEM) x U^T terms (shared memory), K = 64
        {
          constexpr uint32_t idesc = tc::idesc_bf16(kOM, 32);
          constexpr int np = (NT == 2) ? 3 : 6;
          constexpr int pa[6] = {NT == 2 ? 1 : 2, NT == 2 ? 0 : 1, 0, 1, 0, 0};
          constexpr int pb[6] = {0, 1, NT == 2 ? 0 : 2, 0, 1, 0};
          for (int i = 0; i < nt; ++i) {
            const int g = g0 + i, b = g & 1;
            const uint32_t gp = (uint32_t)((g >> 1) & 1);
            if (!wait(&utfull[b], gp)) break;
            if (!wait(&afull[b], gp)) break;
            if (!wait(&cempty[b], gp ^ 1u)) break;
            tc::fence_after_sync();
            const uint64_t ub = ut_desc0 + (uint64_t)(b * (3 * kOUtBox / 16));
            const uint32_t dacc = tmem + kOTmPAcc + 32 * b, abuf = tmem + kOTmABuf + 96 * b;
#pragma unroll
            for (int p = 0; p < np; ++p) {
#pragma unroll
              for (int kk = 0; kk < kON / 16; ++kk)
                tc::mma_bf16_ta(dacc, abuf + 32 * pa[p] + 8 * kk, ub + (uint64_t)((pb[p] * kOUtBox + 32 * kk) / 16),
                                idesc, (p | kk) ? 1u : 0u);
            }
            tc::mma_commit(&mdone[b]);
          }
        }
        // phase 2: D = Pc U^T (A = Pc planes, B = U planes), K = 32
        if (wait(&pcfull, (uint32_t)(k & 1)) && wait(&dinit, (uint32_t)(k & 1))) {
          tc::fence_after_sync();
          constexpr int np = (NPL == 1) ? 3 : 6;
          constexpr int pa[6] = {NPL == 1 ? 1 : 2, NPL == 1 ? 0 : 1, 0, 1, 0, 0};
          constexpr int pb[6] = {0, 1, NPL == 1 ? 0 : 2, 0, 1, 0};
          for (int grp = 0; grp < ngroups; ++grp) {
            if (!wait(&ufull[grp], (uint32_t)(k & 1))) break;
            tc::fence_after_sync();
            const int ntile = grp == 0 ? (nt < kOGroupTiles ? nt : kOGroupTiles) : nt - kOGroupTiles;
            const uint32_t idesc = tc::idesc_bf16(kOM, kON * ntile);
            const uint64_t b0 = u_desc0 + (uint64_t)((grp == 1 && kGroupsApart) ? NPL * kOUGroup / 16 : 0);
            // added onto alpha W: tiles 0-3 in tensor-memory columns 256-511, tiles 4-7 in
            // their homes (columns 0-255)
            const uint32_t d = grp == 0 ? tmem + kOTmD : tmem + kOTmHome;
#pragma unroll
            for (int p = 0; p < np; ++p) {
              const int ao = ((pa[p] >> 1) * kOAPlane + 64 * (pa[p] & 1)) / 16;
              const int bo = ((pb[p] >> 1) * kOUGroup + 64 * (pb[p] & 1)) / 16;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                tc::mma_bf16(d, pc_desc + (uint64_t)(ao + 2 * kk), b0 + (uint64_t)(bo + 2 * kk), idesc, 1u);
            }
            tc::mma_commit(&dfull[grp]);
          }
        }
      }
    }
  } else {
    // ======================= workers (warps 0-7): thread = row, 32 columns =======================
    const float alpha = (float)(1.0 / sqrt((double)a.sigma[0]));
    unsigned int nbar = 0;   // grid barriers passed (thread 0)
    // Grid-wide barrier (thread 0 of each CTA): always arrives, so that a CTA that has given
    // up still releases the others; waits only while nothing has failed.
    // The CTA's writes are ordered before thread 0's release by the named barrier that
    // precedes every call (the cooperative-groups grid-sync pattern).
    auto grid_barrier = [&]() {
      ++nbar;
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.grid_counter) : "memory");
      if (failed) return;
      const long long t0 = clock64();
      while (ld_acquire_u32(P.grid_counter) < nbar * G)
        if (clock64() - t0 > kOWait) {
          failed = 1;
          set_status(status, GIFT_ERR_TIMEOUT);
          return;
        }
    };
    for (int k = 0; k < P.nb; ++k) {
      // the thread's coordinates are re-derived for every tensor from opaque copies, so that
      // the addresses computed from them are not all held live across the batch loop
      int tid_k = tid, r0_k = r0, cb0_k = cb0;
      uint32_t tmem_k = tmem;
      asm volatile("" : "+r"(tid_k), "+r"(r0_k), "+r"(cb0_k), "+r"(tmem_k));
      const int warp = tid_k >> 5, lane = tid_k & 31, quarter = warp & 3, half = warp >> 2;
      const int lr = quarter * 32 + lane, row = r0_k + lr;
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      auto d_slot = [&](int i) {
        return tmem_k + lane_off +
               ((i < kOSmemHomes) ? kOTmD + (uint32_t)(64 * i) : kOTmHome + (uint32_t)(64 * (i - kOSmemHomes))) +
               (uint32_t)(32 * half);
      };
      uint8_t *const stg = sm + kOffCodes;
      const LrEncodeItem &it = P.item[k];
      const uint32_t kp = (uint32_t)(k & 1);
      const int g0 = k * nt;

      // ---------------- phase 1: projection ----------------
      float accp[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) accp[j] = 0.0f;
      auto fold = [&](int g) {
        const int c = g & 1;
        wait(&mdone[c], (uint32_t)((g >> 1) & 1));
        tc::fence_after_sync();
        uint32_t raw[16];
        tc::tmem_ld16_nowait(tmem_k + lane_off + kOTmPAcc + 32 * c + 16 * half, raw);
        tc::tmem_wait_ld16(raw);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&cempty[c]);
#pragma unroll
        for (int q = 0; q < 16; ++q) accp[q] = __fadd_rn(accp[q], __uint_as_float(raw[q]));
      };
      for (int i = 0; i < nt; ++i) {
        const int g = g0 + i, b = g & 1;
        wait(&wfull[i], kp);
        wait(&mdone[b], (uint32_t)(((g >> 1) & 1) ^ 1));
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
        for (int q = 0; q < 16; ++q) tc::bf16_split3x2(x[2 * q], x[2 * q + 1], w1[q], w2[q], w3[q]);
        const uint32_t abase = tmem_k + lane_off + kOTmABuf + 96 * b + 16 * half;
        tc::tmem_st16(abase, w1);
        tc::tmem_st16(abase + 32, w2);
        if (NT == 3) tc::tmem_st16(abase + 64, w3);
        if (i >= kOSmemHomes) {
          uint32_t aw[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) aw[q] = __float_as_uint(__fmul_rn(alpha, x[q]));
          const uint32_t home = tmem_k + lane_off + kOTmHome + (uint32_t)(64 * (i - kOSmemHomes) + 32 * half);
          tc::tmem_st16(home, aw);
          tc::tmem_st16(home + 16, aw + 16);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();   // staging is refilled by TMA
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&afull[b]);
          if (i >= kOSmemHomes) tc::mbar_arrive(&sdone[i - kOSmemHomes]);
        }
        if (i > 0) fold(g - 1);
      }
      fold(g0 + nt - 1);
      if (row < d_out) {
        float4 *dst = reinterpret_cast<float4 *>(P.part + ((size_t)jc * d_out + row) * 32 + 16 * half);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(accp[4 * q], accp[4 * q + 1], accp[4 * q + 2], accp[4 * q + 3]);
      }
      tc::named_bar_sync(1, 32 * kOWarps);
      if (tid_k == 0) grid_barrier();
      tc::named_bar_sync(1, 32 * kOWarps);

      // ---------------- this CTA's share of Pc (rows of its row block) ----------------
      {
        const int ra = r0_k + (kOM * jc) / P.cpr, rz = r0_k + (kOM * (jc + 1)) / P.cpr;
        for (int item = tid_k; item < (rz - ra) * 16; item += 32 * kOWarps) {
          const int rr = ra + (item >> 4), kb = 2 * (item & 15);
          if (rr >= d_out) continue;
          float sum[2] = {0.f, 0.f}, comp[2] = {0.f, 0.f};
          for (int q0 = 0; q0 < P.cpr; q0 += 16) {
            float2 xs2[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
              if (q0 + u < P.cpr)
                xs2[u] = __ldcg(reinterpret_cast<const float2 *>(P.part + ((size_t)(q0 + u) * d_out + rr) * 32 + kb));
#pragma unroll
            for (int u = 0; u < 16; ++u)
              if (q0 + u < P.cpr) {
                const float xs[2] = {xs2[u].x, xs2[u].y};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float y = __fsub_rn(xs[e], comp[e]);
                  const float t = __fadd_rn(sum[e], y);
                  comp[e] = __fsub_rn(__fsub_rn(t, sum[e]), y);
                  sum[e] = t;
                }
              }
          }
          float pc[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) pc[e] = (float)(coef[kb + e] * ((double)sum[e] - (double)comp[e]));
          *reinterpret_cast<float2 *>(P.Pc + (size_t)rr * 32 + kb) = make_float2(pc[0], pc[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) tc::write_term_planes(P.pc_planes, (size_t)d_out, (size_t)rr, kb + e, pc[e], NPL);
        }
      }
      fence_proxy_async_global();   // the planes are read back by TMA
      tc::named_bar_sync(1, 32 * kOWarps);
      if (tid_k == 0) {
        grid_barrier();
        tc::mbar_arrive(&go2);
      }
      // alpha W of the shared-memory tiles into their tensor-memory accumulators (columns
      // 256-511, free since the last fold) while the Pc planes are fetched: phase 2 adds Pc U^T
      // onto them as onto the tensor-memory tiles, and the shared-memory homes are free for
      // the next tensor's tiles from here on
      for (int i = 0; i < nt && i < kOSmemHomes; ++i) {
        const uint8_t *box = sm + kOffHome + i * kOTile + half * kOBox;
        uint32_t aw[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = *reinterpret_cast<const float4 *>(box + sw(lr, c));
          aw[4 * c + 0] = __float_as_uint(__fmul_rn(alpha, v.x));
          aw[4 * c + 1] = __float_as_uint(__fmul_rn(alpha, v.y));
          aw[4 * c + 2] = __float_as_uint(__fmul_rn(alpha, v.z));
          aw[4 * c + 3] = __float_as_uint(__fmul_rn(alpha, v.w));
        }
        tc::tmem_st16(d_slot(i), aw);
        tc::tmem_st16(d_slot(i) + 16, aw + 16);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();   // the homes are refilled by TMA
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&dinit);
        tc::mbar_arrive(&hfree);
      }

      // ---------------- phase 2: CTA amax of W~ (the next tile's load in flight) ----------------
      uint32_t m_run = 0;
      uint32_t nxt[32];
      wait(&dfull[0], kp);
      tc::fence_after_sync();
      tc::tmem_ld32_nowait(d_slot(0), nxt);
      for (int i = 0; i < nt; ++i) {
        const int c0 = (cb0_k + i) * kON;
        tc::tmem_wait_ld(nxt);
        uint32_t raw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = nxt[e];
        if (i + 1 < nt) {
          if (i + 1 == kOGroupTiles) {
            wait(&dfull[1], kp);
            tc::fence_after_sync();
          }
          tc::tmem_ld32_nowait(d_slot(i + 1), nxt);
        }
        if (row < d_out && (c0 + 32 * half) < d_in) {
#pragma unroll
          for (int e = 0; e < 32; ++e) m_run = max(m_run, raw[e] & 0x7FFFFFFFu);
          if (TOUT && it.tout) {
            float4 *dst = reinterpret_cast<float4 *>(it.tout + (size_t)row * d_in + c0 + 32 * half);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_float4(__uint_as_float(raw[4 * c]), __uint_as_float(raw[4 * c + 1]),
                                   __uint_as_float(raw[4 * c + 2]), __uint_as_float(raw[4 * c + 3]));
          }
        }
      }
      m_run = warp_max_u32(m_run);
      if (lane == 0) red[warp] = m_run;
      tc::fence_before_sync();
      tc::named_bar_sync(1, 32 * kOWarps);
      tc::fence_after_sync();
      if (EPI == LR_AMAX) {
        // amax only: max-accumulated into the caller's word, no pack
        if (tid_k == 0) {
          uint32_t m = 0;
          for (int w = 0; w < kOWarps; ++w) m = max(m, red[w]);
          if (m > 0x7F7FFFFFu) set_status(status, GIFT_ERR_NONFINITE);
          if (m) asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(it.amax_out), "r"(m) : "memory");
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sfree);
        continue;
      }
      if (tid_k == 0) {
        uint32_t m = 0;
        for (int w = 0; w < kOWarps; ++w) m = max(m, red[w]);
        float amax;
        if (it.amax_in) {
          amax = it.amax_in[0];
        } else {
          unsigned int *word = reinterpret_cast<unsigned int *>(a.amax_ws) + k;
          // no return value needed: ordered before the barrier's release by program order
          if (m) asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(word), "r"(m) : "memory");
          grid_barrier();
          amax = __uint_as_float(ld_acquire_u32(word));
        }
        amax_sh = amax;
        if (blockIdx.x == 0) {
          if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
          if (EPI == LR_PACK_TENSOR) reinterpret_cast<float *>(it.scales)[0] = scale_pair(amax, fmax_of<F>()).s;
          else it.tscale[0] = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
          if (it.amax_out) it.amax_out[0] = amax;
        }
      }
      tc::named_bar_sync(1, 32 * kOWarps);
      const float amax = amax_sh;
      const ScalePair sp = scale_pair(amax, fmax_of<F>());
      const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);

      // ---------------- phase 3: pack out of tensor memory (next tile's load in flight) ----------------
      tc::tmem_ld32_nowait(d_slot(0), nxt);
      for (int i = 0; i < nt; ++i) {
        tc::tmem_wait_ld(nxt);
        uint32_t raw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = nxt[e];
        if (i + 1 < nt) tc::tmem_ld32_nowait(d_slot(i + 1), nxt);
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
        if (EPI == LR_PACK_TENSOR) {
          uint32_t w4[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const float *x = v + 4 * h;
            w4[h] = pack4_fp8<F>(__fmul_rn(x[0], sp.m), __fmul_rn(x[1], sp.m), __fmul_rn(x[2], sp.m),
                                 __fmul_rn(x[3], sp.m));
          }
          const int c = 4 * i + 2 * half;   // 16-byte chunk of the CTA's 512-byte code row
          *reinterpret_cast<uint4 *>(stg + stg8(lr, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          *reinterpret_cast<uint4 *>(stg + stg8(lr, c + 1)) = make_uint4(w4[4], w4[5], w4[6], w4[7]);
        } else {
          uint16_t sc = 0;
          uint32_t cw[4];
#pragma unroll
          for (int gq = 0; gq < 2; ++gq) {
            uint32_t gm = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) gm = max(gm, abs_bits(v[16 * gq + e]));
            const Nv4Group grp = nvfp4_group(__uint_as_float(gm), s_t);
            float y[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) y[e] = __fmul_rn(v[16 * gq + e], grp.r);
            cw[2 * gq] = pack8_e2m1(y);
            cw[2 * gq + 1] = pack8_e2m1(y + 8);
            sc |= (uint16_t)grp.e_code << (8 * gq);
          }
          *reinterpret_cast<uint4 *>(stg + stg4(lr, 2 * i + half)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t *>(stg + kOStgScales + lr * 32 + 4 * i + 2 * half) = sc;
        }
      }
      // every worker's tensor-memory reads of this tensor are done past this barrier (the next
      // tensor's phase 1 writes those columns), and the code rows are complete
      tc::fence_before_sync();
      tc::named_bar_sync(1, 32 * kOWarps);
      tc::fence_after_sync();
      // coalesced copy-out of the CTA's code rows (and NVFP4 block scales)
      const int cbase = cb0_k * kON;
      if (EPI == LR_PACK_TENSOR) {
        for (int r = warp; r < kOM; r += kOWarps) {
          const int gr = r0_k + r, col = cbase + 16 * lane;
          if (gr < d_out && lane < 4 * nt && col < d_in)
            *reinterpret_cast<uint4 *>(it.codes + (size_t)gr * d_in + col) = *reinterpret_cast<const uint4 *>(stg + stg8(r, lane));
        }
      } else {
        for (int item = tid_k; item < kOM * 16; item += 32 * kOWarps) {
          const int r = item >> 4, c = item & 15, gr = r0_k + r, col = cbase + 32 * c;
          if (gr < d_out && c < 2 * nt && col < d_in)
            *reinterpret_cast<uint4 *>(it.codes + (((size_t)gr * d_in + col) >> 1)) = *reinterpret_cast<const uint4 *>(stg + stg4(r, c));
        }
        for (int item = tid_k; item < kOM * 16; item += 32 * kOWarps) {
          const int r = item >> 4, q = item & 15, gr = r0_k + r, col = cbase + 32 * q;   // two scale bytes per 32 columns
          if (gr < d_out && q < 2 * nt && col < d_in)
            *reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(it.scales) + (size_t)gr * (d_in / kNvGroup) + col / kNvGroup) =
                *reinterpret_cast<const uint16_t *>(stg + kOStgScales + r * 32 + 2 * q);
        }
      }
      // the staging region is refilled by TMA (the next tensor's staging tiles)
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sfree);
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
cudaError_t onepass_launch(const Launch &L, const OnePassParams &P, const OnePassMaps &M, int grid) {
  const LrApply &a = P.a;
  const LrPlanes pl = lr_planes(a.split, a.d_out, a.d_in);
  constexpr int NPL = NT - 1;
  CUtensorMap tmUT, tmU, tmPc;
  if (!omap(&tmUT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.ut_planes, 96, (uint64_t)a.d_in, kON, 32) ||
      !omap(&tmU, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.u_planes, (uint64_t)NPL * a.d_in, 32, 32, kOGroupTiles * kON) ||
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
  return cudaLaunchKernelEx(&cfg, kern, P, M, tmUT, tmU, tmPc, L.status);
}

template <int NT>
cudaError_t onepass_dispatch(const Launch &L, int epi, int fmt, const OnePassParams &P, const OnePassMaps &M,
                             int grid, bool t) {
  if (epi == LR_AMAX) return onepass_launch<LR_AMAX, FMT_E4M3, NT, false>(L, P, M, grid);
  if (epi == LR_NVFP4)
    return t ? onepass_launch<LR_NVFP4, FMT_E4M3, NT, true>(L, P, M, grid)
             : onepass_launch<LR_NVFP4, FMT_E4M3, NT, false>(L, P, M, grid);
  if (fmt == GIFT_FMT_E5M2)
    return t ? onepass_launch<LR_PACK_TENSOR, FMT_E5M2, NT, true>(L, P, M, grid)
             : onepass_launch<LR_PACK_TENSOR, FMT_E5M2, NT, false>(L, P, M, grid);
  return t ? onepass_launch<LR_PACK_TENSOR, FMT_E4M3, NT, true>(L, P, M, grid)
           : onepass_launch<LR_PACK_TENSOR, FMT_E4M3, NT, false>(L, P, M, grid);
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

// U planes (and the zeroed counters) must be in a.split, a.amax_ws[0..nb) zero for the
// tensors without a caller amax, a.grid_counter zero.  The items' W replace a.X (each must
// pass lr_encode_onepass_ok in a.X's place); a's per-tensor outputs are ignored.
cudaError_t launch_lr_encode_onepass_batch(const Launch &L, int epi, int fmt, const LrApply &a, const float *mu,
                                           float *part, float *Pc, int nb, const LrEncodeItem *items) {
  if (nb < 1 || nb > kOnePassMaxBatch) return cudaErrorInvalidValue;
  int cpr = 0;
  const int grid = onepass_plan(L.sms, a.d_out, a.d_in, &cpr);
  if (grid <= 0) return cudaErrorInvalidValue;
  OnePassParams P;
  std::memset(&P, 0, sizeof(P));
  P.a = a;
  P.mu = mu;
  P.tiles_n = (a.d_in + kON - 1) / kON;
  P.cpr = cpr;
  P.nb = nb;
  P.part = part;
  P.Pc = Pc;
  P.pc_planes = lr_planes(a.split, a.d_out, a.d_in).pc;
  P.grid_counter = a.grid_counter;
  OnePassMaps M;
  std::memset(&M, 0, sizeof(M));
  bool tout = false;
  for (int k = 0; k < nb; ++k) {
    P.item[k] = items[k];
    tout = tout || items[k].tout != nullptr;
    if (!omap(&M.w[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, items[k].X, (uint64_t)a.d_out, (uint64_t)a.d_in, 32, kOM))
      return cudaErrorInvalidValue;
  }
  return a.terms == 1 ? onepass_dispatch<2>(L, epi, fmt, P, M, grid, tout)
                      : onepass_dispatch<3>(L, epi, fmt, P, M, grid, tout);
}

cudaError_t launch_lr_encode_onepass(const Launch &L, int epi, int fmt, const LrApply &a, const float *mu,
                                     float *part, float *Pc) {
  LrEncodeItem it;
  it.X = a.X;
  it.codes = a.codes;
  it.scales = a.scales;
  it.tscale = a.tscale;
  it.amax_out = a.amax_out;
  it.tout = a.tout;
  it.amax_in = a.amax_in;
  return launch_lr_encode_onepass_batch(L, epi, fmt, a, mu, part, Pc, 1, &it);
}

}  // namespace gift
