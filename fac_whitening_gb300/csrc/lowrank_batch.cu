// Rank-r encode of a batch of tensors that share the factor (the data-parallel replicas of a
// layer's gradient) in two streaming passes plus a small reduce.
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17): W~ = sigma^-1/2 W +
// ((W U) diag(c)) U^T, c = mu^-1/2 - sigma^-1/2, then the per-tensor amax scale and the FP8
// (or NVFP4) pack.
//
// CTA = one 128-row block x at most 8 column tiles of 64 (the same decomposition in both
// passes, so a CTA's U planes are the same for every tensor of the batch).
//   pass A (k_lr_proj_batch): P = W U for every tensor.  The W tiles stream through a 4-deep
//          TMA ring, the U^T term planes of the CTA's columns stay in shared memory for the whole
//          batch.  Eight warps split each tile exactly into BF16 terms (tensor-memory A
//          operand, 2 buffers; 3 accumulators, each folded two tiles after its MMAs were
//          issued); one thread issues per K step three MMAs whose B operands are
//          the stacked U^T terms ([u1;u2;u3], [u1;u2], [u1]), so that the six products
//          x_i u_j (i + j <= 2) land in three 32-column groups of a fresh accumulator per tile;
//          the groups are added and folded into the slice sum with round-to-nearest FP32 adds.
//   reduce (k_lr_pc_batch): Pc / alpha = (c / alpha) * (sum over the slices, slice order,
//          compensated FP32; c / alpha = (sigma / mu)^1/2 - 1 in FP64), as BF16 term planes.
//   pass B (k_lr_apply_batch, cooperative): D = W + (Pc / alpha) U^T of the whole CTA block
//          in tensor memory (8 tiles x 64 columns), W~ = alpha D.  The W tiles stream through a
//          3-deep TMA ring and the tensor core copies them into tensor memory (tcgen05.cp);
//          two N = 256 MMA chains add (Pc / alpha) U^T; the workers take the amax of alpha D,
//          one clock-bounded grid barrier gives the tensor amax, and the pack reads tensor
//          memory and stores the codes through shared memory as coalesced rows.  A group of
//          tensor memory takes the next tensor's W as soon as its codes are packed, the next
//          tensor's first tiles already waiting in the ring; its Pc and U planes load as soon
//          as this tensor's MMAs are done.  The tensors are taken last to first: the last
//          ones pass A read are still in L2.
// W is read twice (pass A and pass B) but neither pass waits on the other tensors.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kBM = 128, kBN = 64;
constexpr int kBMaxTiles = 8;
constexpr int kBWarps = 8;
constexpr int kBThreads = 32 * (kBWarps + 2);
constexpr int kBBox = 128 * 128;        // 128 rows x 32 FP32 (one TMA box of W)
constexpr int kBTile = 2 * kBBox;       // 32 KB: a 128 x 64 tile of W
constexpr int kBStages = 4;             // W ring
constexpr int kBUtPlane = 32 * 128;     // U^T term plane of a tile: 32 rows x 64 BF16
constexpr int kBGroupTiles = 4;         // pass B: tiles per MMA group (N = 256)
constexpr int kBUGroup = kBGroupTiles * kBN * 128;   // U plane box of a group: 256 rows x 128 B
constexpr int kBPcPlane = 128 * 128;    // Pc plane box: 128 rows x 128 B
constexpr long long kBWait = 4000000000LL;

// pass A shared memory: the U^T planes of the CTA's tiles, then the W ring
constexpr int kAOffUt = 0;
constexpr int kAOffStage = kBMaxTiles * 3 * kBUtPlane;                // 96 KB
constexpr int kASmem = kAOffStage + kBStages * kBTile;                // 224 KB
// pass B shared memory: a 3-deep W ring, the Pc planes, a group's U planes, code staging
constexpr int kBRing = 3;
constexpr int kBOffPc = kBRing * kBTile;                              // 96 KB
constexpr int kBOffU = kBOffPc + 2 * kBPcPlane;                       // 128 KB
constexpr int kBOffStg = kBOffU + 2 * kBUGroup;                       // 192 KB
constexpr int kBStg = 128 * 256;                                      // a group's FP8 code rows
constexpr int kBSmem = kBOffStg + kBStg;                              // 224 KB
constexpr int kBOffScales = 128 * 128;   // NVFP4 staging: block scales after the code rows

struct ProjBatchParams {
  int d_out, d_in, tiles_n, cpr, nb;
  float *part;   // nb x cpr x d_out x 32 slice partials
};
struct BatchMaps {
  CUtensorMap w[kEncodeBatchMax];   // W of each tensor
};
struct ApplyBatchParams {
  LrApply a;                 // factor, planes, shapes; a.amax_ws = one word per tensor
  int tiles_n, cpr, nb;
  int reverse;               // take the tensors last to first (the last ones projected are still in L2)
  unsigned int *grid_counter;   // zero on entry
  LrEncodeItem item[kEncodeBatchMax];
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int sw(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }
// code staging of one group of four tiles: FP8 rows of 16 x 16 bytes, NVFP4 rows of 8 x 16
// bytes, 16-byte chunks XOR-swizzled by row; NVFP4 block scales 16 bytes per row after them
__device__ __forceinline__ int stg8(int r, int c) { return r * 256 + ((c ^ (r & 15)) << 4); }
__device__ __forceinline__ int stg4(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// The CTA's block: row block rb, column slice jc of the row block's tiles.
struct BlockOf {
  int rb, jc, cb0, nt, r0;
};
__device__ __forceinline__ BlockOf block_of(int tiles_n, int cpr) {
  BlockOf b;
  b.rb = blockIdx.x / cpr;
  b.jc = blockIdx.x - b.rb * cpr;
  b.cb0 = (int)(((long long)tiles_n * b.jc) / cpr);
  b.nt = (int)(((long long)tiles_n * (b.jc + 1)) / cpr) - b.cb0;   // 1..8
  b.r0 = b.rb * kBM;
  return b;
}

}  // namespace

// ---------------------------------------------------------------------------------------
// pass A: slice partials of P = W U for every tensor of the batch
template <int NT>
__global__ void __launch_bounds__(kBThreads, 1) k_lr_proj_batch(const __grid_constant__ ProjBatchParams P,
                                                                const __grid_constant__ BatchMaps M,
                                                                const __grid_constant__ CUtensorMap tmUT,
                                                                int *status) {
  constexpr int kABufs = 2;                       // A operand buffers
  constexpr int kDBufs = 3;                       // accumulators: a tile is folded two tiles later
  constexpr int ACOLS = 32 * NT;                  // A buffer: NT terms x 64 BF16 of K
  constexpr int DCOLS = 32 * NT;                  // accumulator: one 32-column group per U term
  constexpr uint32_t kTmD = kABufs * ACOLS;       // accumulators after the A buffers
  static_assert(kTmD + kDBufs * DCOLS <= 512, "tensor memory");
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t utfull, sfull[kBStages], sempty[kBStages], afull[kABufs], aempty[kABufs], cfull[kDBufs],
      cempty[kDBufs];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = P.d_out;
  const BlockOf B = block_of(P.tiles_n, P.cpr);
  const int nt = B.nt, total = P.nb * nt;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    tc::mbar_init(&utfull, 1);
    for (int s = 0; s < kBStages; ++s) {
      tc::mbar_init(&sfull[s], 1);
      tc::mbar_init(&sempty[s], kBWarps);
    }
    for (int a = 0; a < kABufs; ++a) {
      tc::mbar_init(&afull[a], kBWarps);
      tc::mbar_init(&aempty[a], 1);
    }
    for (int c = 0; c < kDBufs; ++c) {
      tc::mbar_init(&cfull[c], 1);
      tc::mbar_init(&cempty[c], kBWarps);
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
    if (!tc::mbar_wait_bounded(bar, parity, kBWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kBWarps) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tc::prefetch_tensormap(&tmUT);
      for (int k = 0; k < P.nb; ++k) tc::prefetch_tensormap(&M.w[k]);
      tc::mbar_arrive_expect_tx(&utfull, nt * NT * kBUtPlane);
      for (int i = 0; i < nt; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t)
          tc::tma_load_2d(sm + kAOffUt + (i * NT + t) * kBUtPlane, &tmUT, (B.cb0 + i) * kBN, 32 * t, &utfull);
      for (int g = 0; g < total; ++g) {
        const int k = g / nt, i = g - k * nt, s = g & (kBStages - 1);
        if (g >= kBStages && !wait(&sempty[s], (uint32_t)(((g / kBStages) - 1) & 1))) break;
        uint8_t *dst = sm + kAOffStage + s * kBTile;
        tc::mbar_arrive_expect_tx(&sfull[s], kBTile);
        tc::tma_load_2d(dst, &M.w[k], (B.cb0 + i) * kBN, B.r0, &sfull[s]);
        tc::tma_load_2d(dst + kBBox, &M.w[k], (B.cb0 + i) * kBN + 32, B.r0, &sfull[s]);
      }
    }
  } else if (warp == kBWarps + 1) {
    // ======================= MMA issuer =======================
    if (lane == 0 && wait(&utfull, 0)) {
      tc::fence_after_sync();
      const uint64_t ut0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kAOffUt));
      constexpr uint32_t id1 = tc::idesc_bf16(kBM, 32 * NT);         // x1 . [u1; ...; u_NT]
      constexpr uint32_t id2 = tc::idesc_bf16(kBM, 32 * (NT - 1));   // x2 . [u1; ...]
      constexpr uint32_t id3 = tc::idesc_bf16(kBM, 32);              // x3 . u1
      for (int g = 0; g < total; ++g) {
        const int i = g % nt, a = g % kABufs, c = g % kDBufs;
        if (!wait(&afull[a], (uint32_t)((g / kABufs) & 1))) break;
        if (!wait(&cempty[c], (uint32_t)(((g / kDBufs) & 1) ^ 1))) break;
        tc::fence_after_sync();
        const uint64_t ub = ut0 + (uint64_t)(i * NT * kBUtPlane / 16);   // the tile's stacked U^T terms
        const uint32_t d = tmem + kTmD + DCOLS * c, ab = tmem + ACOLS * a;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // the first MMA writes every column group, so it opens the accumulator
          tc::mma_bf16_ta(d, ab + 8 * kk, ub + (uint64_t)(2 * kk), id1, kk ? 1u : 0u);
          tc::mma_bf16_ta(d, ab + 32 + 8 * kk, ub + (uint64_t)(2 * kk), id2, 1u);
          if (NT == 3) tc::mma_bf16_ta(d, ab + 64 + 8 * kk, ub + (uint64_t)(2 * kk), id3, 1u);
        }
        tc::mma_commit(&aempty[a]);
        tc::mma_commit(&cfull[c]);
      }
    }
  } else {
    // ======================= workers (warps 0-7): thread = row, 32 columns =======================
    const int quarter = warp & 3, half = warp >> 2;
    const int lr = quarter * 32 + lane, row = B.r0 + lr;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float accp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) accp[j] = 0.0f;
    // fold tile g's accumulator into the slice sum; after a tensor's last tile, write the slice
    auto fold = [&](int g) {
      const int c = g % kDBufs;
      wait(&cfull[c], (uint32_t)((g / kDBufs) & 1));
      tc::fence_after_sync();
      const uint32_t base = tmem + lane_off + kTmD + DCOLS * c + 16 * half;
      uint32_t d0[16], d1[16], d2[16];
      tc::tmem_ld16_nowait(base, d0);
      tc::tmem_ld16_nowait(base + 32, d1);
      if (NT == 3) tc::tmem_ld16_nowait(base + 64, d2);
      tc::tmem_wait_ld16(d0);
      tc::tmem_wait_ld16(d1);
      if (NT == 3) tc::tmem_wait_ld16(d2);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&cempty[c]);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        float t = __fadd_rn(__uint_as_float(d1[q]), __uint_as_float(d0[q]));
        if (NT == 3) t = __fadd_rn(__fadd_rn(__uint_as_float(d2[q]), __uint_as_float(d1[q])), __uint_as_float(d0[q]));
        accp[q] = __fadd_rn(accp[q], t);
      }
      const int k = g / nt;
      if (g - k * nt == nt - 1) {
        if (row < d_out) {
          float4 *dst = reinterpret_cast<float4 *>(P.part + (((size_t)k * P.cpr + B.jc) * d_out + row) * 32 + 16 * half);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_float4(accp[4 * q], accp[4 * q + 1], accp[4 * q + 2], accp[4 * q + 3]);
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) accp[q] = 0.0f;
      }
    };
    for (int g = 0; g < total; ++g) {
      const int s = g & (kBStages - 1), a = g % kABufs;
      wait(&sfull[s], (uint32_t)((g / kBStages) & 1));
      wait(&aempty[a], (uint32_t)(((g / kABufs) & 1) ^ 1));
      tc::fence_after_sync();
      const uint8_t *box = sm + kAOffStage + s * kBTile + half * kBBox;
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
      const uint32_t abase = tmem + lane_off + ACOLS * a + 16 * half;
      tc::tmem_st16(abase, w1);
      tc::tmem_st16(abase + 32, w2);
      if (NT == 3) tc::tmem_st16(abase + 64, w3);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();   // the ring slot is refilled by TMA
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&sempty[s]);
        tc::mbar_arrive(&afull[a]);
      }
      // fold two tiles behind: that tile's MMAs are long done, so the split of the next tile
      // is not held up by the newest MMAs
      if (g > 1) fold(g - 2);
    }
    for (int g = total - 2; g < total; ++g)
      if (g >= 0) fold(g);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------------
// reduce: Pc / alpha (alpha = sigma^-1/2) of every tensor from its slice partials, written as
// BF16 term planes
template <int NPL>
__global__ void __launch_bounds__(256) k_lr_pc_batch(const float *__restrict__ part, int nb, int cpr, int d_out,
                                                     const float *__restrict__ mu, const float *__restrict__ sigma,
                                                     int rank, uint16_t *pc_planes, int *status) {
  __shared__ double cf[32];   // c_k in FP64, formed once per block
  if (threadIdx.x < 32) {
    const int k = threadIdx.x;
    double c = 0.0;
    if (k < rank) {
      const double m = (double)mu[k], sg = (double)sigma[0];
      if (!(m > 0.0) || !(sg > 0.0)) {
        if (blockIdx.x == 0) set_status(status, GIFT_ERR_NOT_PD);
      } else {
        c = (1.0 / sqrt(m) - 1.0 / sqrt(sg)) * sqrt(sg);   // c / alpha: pass B adds onto W
      }
    }
    cf[k] = c;
  }
  __syncthreads();
  // thread = (tensor, row, 2 consecutive columns); the planes take one 4-byte store per term
  const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per = (long long)d_out * 16;
  if (item >= per * nb) return;
  const int k = (int)(item / per);
  const int rem = (int)(item - (long long)k * per);
  const int row = rem >> 4, kb = 2 * (rem & 15);
  float sum[2] = {0.f, 0.f}, comp[2] = {0.f, 0.f};
  const float *src = part + ((size_t)k * cpr * d_out + row) * 32 + kb;
  for (int q0 = 0; q0 < cpr; q0 += 16) {
    float2 xs2[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (q0 + u < cpr) xs2[u] = __ldcg(reinterpret_cast<const float2 *>(src + (size_t)(q0 + u) * d_out * 32));
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (q0 + u < cpr) {
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
  const float p0 = (float)(cf[kb] * ((double)sum[0] - (double)comp[0]));
  const float p1 = (float)(cf[kb + 1] * ((double)sum[1] - (double)comp[1]));
  uint32_t t1, t2, t3;
  tc::bf16_split3x2(p0, p1, t1, t2, t3);
  // planes of tensor k: plane 0 rows [t1 | t2], plane 1 rows [t3 | 0] (64 BF16 each)
  uint16_t *q = pc_planes + (size_t)k * 2 * d_out * 64 + (size_t)row * 64;
  *reinterpret_cast<uint32_t *>(q + kb) = t1;
  *reinterpret_cast<uint32_t *>(q + 32 + kb) = t2;
  if (NPL > 1) {
    *reinterpret_cast<uint32_t *>(q + (size_t)d_out * 64 + kb) = t3;
    *reinterpret_cast<uint32_t *>(q + (size_t)d_out * 64 + 32 + kb) = 0u;
  }
}

// ---------------------------------------------------------------------------------------
// pass B: D = W + (Pc / alpha) U^T held in tensor memory, W~ = alpha D, tensor amax, pack
template <int EPI, int F, int NPL, bool TOUT>
__global__ void __launch_bounds__(kBThreads, 1) k_lr_apply_batch(const __grid_constant__ ApplyBatchParams P,
                                                                 const __grid_constant__ BatchMaps M,
                                                                 const __grid_constant__ CUtensorMap tmU,
                                                                 const __grid_constant__ CUtensorMap tmPc,
                                                                 int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  // per-tensor barriers complete once per tensor (parity = tensor & 1); the ring counts tiles
  // across the batch
  // hfree[grp]: the previous tensor's codes of group grp are packed, its tensor memory is free
  __shared__ uint64_t sfull[kBRing], sempty[kBRing], pcfull, ufull[2], hfree[2], dfull[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[kBWarps];
  __shared__ float amax_sh;
  __shared__ volatile int failed;

  const LrApply &a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = a.d_out, d_in = a.d_in;
  const BlockOf B = block_of(P.tiles_n, P.cpr);
  const int nt = B.nt;
  const int ngroups = nt > kBGroupTiles ? 2 : 1;
  const int ntile0 = nt < kBGroupTiles ? nt : kBGroupTiles;   // tiles of the first group
  const unsigned int G = gridDim.x;
  auto tix = [&](int k) { return P.reverse ? P.nb - 1 - k : k; };   // tensor at position k

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kBRing; ++s) {
      tc::mbar_init(&sfull[s], 1);
      tc::mbar_init(&sempty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(&ufull[k], 1);
      tc::mbar_init(&hfree[k], kBWarps);
      tc::mbar_init(&dfull[k], 1);
    }
    tc::mbar_init(&pcfull, 1);
    tc::fence_mbar_init();
    failed = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (failed) return false;
    if (!tc::mbar_wait_bounded(bar, parity, kBWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kBWarps) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tc::prefetch_tensormap(&tmU);
      tc::prefetch_tensormap(&tmPc);
      for (int k = 0; k < P.nb; ++k) tc::prefetch_tensormap(&M.w[k]);
      auto load_w = [&](int k, int i) {
        const int g = k * nt + i, s = g % kBRing;
        if (g >= kBRing && !wait(&sempty[s], (uint32_t)(((g / kBRing) - 1) & 1))) return false;
        uint8_t *dst = sm + s * kBTile;
        tc::mbar_arrive_expect_tx(&sfull[s], kBTile);
        const CUtensorMap *mw = &M.w[tix(k)];
        tc::tma_load_2d(dst, mw, (B.cb0 + i) * kBN, B.r0, &sfull[s]);
        tc::tma_load_2d(dst + kBBox, mw, (B.cb0 + i) * kBN + 32, B.r0, &sfull[s]);
        return true;
      };
      // a group's U planes: one 256-row box per plane (rows past the CTA's tiles unused)
      auto load_group = [&](int grp) {
        tc::mbar_arrive_expect_tx(&ufull[grp], NPL * kBUGroup);
#pragma unroll
        for (int q = 0; q < NPL; ++q)
          tc::tma_load_2d(sm + kBOffU + q * kBUGroup, &tmU, 0, q * d_in + (B.cb0 + kBGroupTiles * grp) * kBN,
                          &ufull[grp]);
      };
      for (int k = 0; k < P.nb; ++k) {
        const uint32_t kp = (uint32_t)(k & 1), pp = kp ^ 1u;
        // the first group's U planes and the Pc planes as soon as the previous tensor's MMAs
        // are done with their regions, ahead of this tensor's W tiles (which wait for ring
        // slots and queue in the same TMA unit)
        if (k > 0 && !wait(&dfull[ngroups - 1], pp)) break;
        load_group(0);
        tc::mbar_arrive_expect_tx(&pcfull, NPL * kBPcPlane);
#pragma unroll
        for (int q = 0; q < NPL; ++q)
          tc::tma_load_2d(sm + kBOffPc + q * kBPcPlane, &tmPc, 0, (2 * tix(k) + q) * d_out + B.r0, &pcfull);
        bool ok = true;
        for (int i = 0; i < nt && ok; ++i) ok = load_w(k, i);
        if (!ok) break;
        if (ngroups == 2) {
          if (!wait(&dfull[0], kp)) break;   // the first group's MMAs are done with the region
          load_group(1);
        }
      }
    }
  } else if (warp == kBWarps + 1) {
    // ======================= MMA issuer =======================
    // Per group: each W tile is copied from the ring into its tensor-memory home
    // (tcgen05.cp, 8 copies of 128 rows x 32 bytes), then one N = 256 MMA chain adds
    // (Pc / alpha) U^T onto the group's tiles (copies and MMAs run in issue order).
    if (lane == 0) {
      const uint64_t pc0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kBOffPc));
      const uint64_t u0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm + kBOffU));
      const uint64_t w0 = tc::sdesc_kmajor_sw128(tc::smem_u32(sm));
      constexpr int np = (NPL == 1) ? 3 : 6;
      constexpr int pa[6] = {NPL == 1 ? 1 : 2, NPL == 1 ? 0 : 1, 0, 1, 0, 0};
      constexpr int pb[6] = {0, 1, NPL == 1 ? 0 : 2, 0, 1, 0};
      for (int k = 0; k < P.nb && !failed; ++k) {
        const uint32_t kp = (uint32_t)(k & 1), pp = kp ^ 1u;
        for (int grp = 0; grp < ngroups; ++grp) {
          if (k > 0 && !wait(&hfree[grp], pp)) break;   // the previous tensor's codes are out
          const int i0 = kBGroupTiles * grp, i1 = grp == 0 ? ntile0 : nt;
          bool ok = true;
          for (int i = i0; i < i1 && ok; ++i) {
            const int g = k * nt + i, s = g % kBRing;
            if (!(ok = wait(&sfull[s], (uint32_t)((g / kBRing) & 1)))) break;
            tc::fence_after_sync();
            const uint64_t ws = w0 + (uint64_t)(s * kBTile / 16);
#pragma unroll
            for (int h = 0; h < 2; ++h)      // the tile's two 32-column boxes
#pragma unroll
              for (int j = 0; j < 4; ++j)    // 8 columns per copy
                tc::cp_128x256b(tmem + (uint32_t)(kBN * i + 32 * h + 8 * j),
                                ws + (uint64_t)((h * kBBox + 32 * j) / 16));
            tc::mma_commit(&sempty[s]);
          }
          if (!ok || (grp == 0 && !wait(&pcfull, kp)) || !wait(&ufull[grp], kp)) break;
          tc::fence_after_sync();
          const int ntile = i1 - i0;
          const uint32_t idesc = tc::idesc_bf16(kBM, kBN * ntile);
          const uint32_t d = tmem + (uint32_t)(kBN * i0);
#pragma unroll
          for (int p = 0; p < np; ++p) {
            const int ao = ((pa[p] >> 1) * kBPcPlane + 64 * (pa[p] & 1)) / 16;
            const int bo = ((pb[p] >> 1) * kBUGroup + 64 * (pb[p] & 1)) / 16;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              tc::mma_bf16(d, pc0 + (uint64_t)(ao + 2 * kk), u0 + (uint64_t)(bo + 2 * kk), idesc, 1u);
          }
          tc::mma_commit(&dfull[grp]);
        }
      }
    }
  } else {
    // ======================= workers (warps 0-7): thread = row, 32 columns =======================
    const float alpha = (float)(1.0 / sqrt((double)a.sigma[0]));
    unsigned int nbar = 0;   // grid barriers passed (thread 0)
    // Grid-wide barrier (thread 0 of each CTA, after a named barrier of the workers): always
    // arrives, so that a CTA that has given up still releases the others.
    auto grid_barrier = [&]() {
      ++nbar;
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.grid_counter) : "memory");
      if (failed) return;
      const long long t0 = clock64();
      while (ld_acquire_u32(P.grid_counter) < nbar * G)
        if (clock64() - t0 > kBWait) {
          failed = 1;
          set_status(status, GIFT_ERR_TIMEOUT);
          return;
        }
    };
    for (int k = 0; k < P.nb; ++k) {
      // the thread's coordinates are re-derived for every tensor from opaque copies, so that
      // the addresses computed from them are not all held live across the batch loop
      int tid_k = tid, r0_k = B.r0;
      uint32_t tmem_k = tmem;
      asm volatile("" : "+r"(tid_k), "+r"(r0_k), "+r"(tmem_k));
      const int wk = tid_k >> 5, ln = tid_k & 31, quarter = wk & 3, half = wk >> 2;
      const int lr = quarter * 32 + ln, row = r0_k + lr;
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t home0 = tmem_k + lane_off + (uint32_t)(32 * half);
      auto slot = [&](int i) { return home0 + (uint32_t)(kBN * i); };
      const LrEncodeItem &it = P.item[tix(k)];
      const uint32_t kp = (uint32_t)(k & 1);

      // ---------------- W~ = alpha D: amax (and the transformed copy), next tile's load in flight ----------------
      uint32_t m_run = 0;
      uint32_t nxt[32];
      wait(&dfull[0], kp);
      tc::fence_after_sync();
      tc::tmem_ld32_nowait(slot(0), nxt);
      for (int i = 0; i < nt; ++i) {
        const int c0 = (B.cb0 + i) * kBN;
        tc::tmem_wait_ld(nxt);
        uint32_t raw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) raw[e] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(nxt[e])));
        if (i + 1 < nt) {
          if (i + 1 == kBGroupTiles) {
            wait(&dfull[1], kp);
            tc::fence_after_sync();
          }
          tc::tmem_ld32_nowait(slot(i + 1), nxt);
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
      if (ln == 0) red[wk] = m_run;
      tc::fence_before_sync();
      tc::named_bar_sync(1, 32 * kBWarps);
      if (EPI == LR_AMAX) {
        // amax only: max-accumulated into the caller's word, no pack
        if (tid_k == 0) {
          uint32_t m = 0;
          for (int w = 0; w < kBWarps; ++w) m = max(m, red[w]);
          if (m > 0x7F7FFFFFu) set_status(status, GIFT_ERR_NONFINITE);
          if (m) asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(it.amax_out), "r"(m) : "memory");
        }
        // every warp's tensor-memory reads are done (the named barrier above)
        tc::fence_before_sync();
        __syncwarp();
        if (ln == 0) {
          tc::mbar_arrive(&hfree[0]);
          if (ngroups == 2) tc::mbar_arrive(&hfree[1]);
        }
        continue;
      }
      if (tid_k == 0) {
        uint32_t m = 0;
        for (int w = 0; w < kBWarps; ++w) m = max(m, red[w]);
        float amax;
        if (it.amax_in) {
          amax = it.amax_in[0];
        } else {
          unsigned int *word = reinterpret_cast<unsigned int *>(a.amax_ws) + tix(k);
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
      tc::named_bar_sync(1, 32 * kBWarps);
      const float amax = amax_sh;
      const ScalePair sp = scale_pair(amax, fmax_of<F>());
      const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);

      // ---------------- pack, one group of four tiles at a time through the staging region ----------------
      uint8_t *const stg = sm + kBOffStg;
      const int cbase = B.cb0 * kBN;
      for (int grp = 0; grp < ngroups; ++grp) {
        const int i0 = kBGroupTiles * grp, i1 = grp == 0 ? ntile0 : nt;
        tc::tmem_ld32_nowait(slot(i0), nxt);
        for (int i = i0; i < i1; ++i) {
          const int j = i - i0;   // tile within the group
          tc::tmem_wait_ld(nxt);
          uint32_t raw[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) raw[e] = nxt[e];
          if (i + 1 < i1) tc::tmem_ld32_nowait(slot(i + 1), nxt);
          if (i + 1 == i1) {
            // this warp's reads of the group are done: the tensor memory takes the next
            // tensor's W
            tc::fence_before_sync();
            __syncwarp();
            if (ln == 0) tc::mbar_arrive(&hfree[grp]);
          }
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __fmul_rn(alpha, __uint_as_float(raw[e]));
          if (EPI == LR_PACK_TENSOR) {
            uint32_t w4[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float *x = v + 4 * h;
              w4[h] = pack4_fp8<F>(__fmul_rn(x[0], sp.m), __fmul_rn(x[1], sp.m), __fmul_rn(x[2], sp.m),
                                   __fmul_rn(x[3], sp.m));
            }
            const int c = 4 * j + 2 * half;   // 16-byte chunk of the group's 256-byte code row
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
              const Nv4Group grpq = nvfp4_group(__uint_as_float(gm), s_t);
              float y[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) y[e] = __fmul_rn(v[16 * gq + e], grpq.r);
              cw[2 * gq] = pack8_e2m1(y);
              cw[2 * gq + 1] = pack8_e2m1(y + 8);
              sc |= (uint16_t)grpq.e_code << (8 * gq);
            }
            *reinterpret_cast<uint4 *>(stg + stg4(lr, 2 * j + half)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            *reinterpret_cast<uint16_t *>(stg + kBOffScales + lr * 16 + 4 * j + 2 * half) = sc;
          }
        }
        // the group's code rows are complete
        tc::named_bar_sync(1, 32 * kBWarps);
        const int gbase = cbase + kBN * i0, ntile = i1 - i0;
        if (EPI == LR_PACK_TENSOR) {
          for (int item = tid_k; item < kBM * 16; item += 32 * kBWarps) {
            const int r = item >> 4, c = item & 15, gr = r0_k + r, col = gbase + 16 * c;
            if (gr < d_out && c < 4 * ntile && col < d_in)
              *reinterpret_cast<uint4 *>(it.codes + (size_t)gr * d_in + col) = *reinterpret_cast<const uint4 *>(stg + stg8(r, c));
          }
        } else {
          for (int item = tid_k; item < kBM * 8; item += 32 * kBWarps) {
            const int r = item >> 3, c = item & 7, gr = r0_k + r, col = gbase + 32 * c;
            if (gr < d_out && c < 2 * ntile && col < d_in)
              *reinterpret_cast<uint4 *>(it.codes + (((size_t)gr * d_in + col) >> 1)) =
                  *reinterpret_cast<const uint4 *>(stg + stg4(r, c));
          }
          for (int item = tid_k; item < kBM * 8; item += 32 * kBWarps) {
            const int r = item >> 3, q = item & 7, gr = r0_k + r, col = gbase + 32 * q;   // two scale bytes per 32 columns
            if (gr < d_out && q < 2 * ntile && col < d_in)
              *reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(it.scales) + (size_t)gr * (d_in / kNvGroup) +
                                            col / kNvGroup) =
                  *reinterpret_cast<const uint16_t *>(stg + kBOffScales + r * 16 + 2 * q);
          }
        }
        // the staging is rewritten by the next group
        tc::named_bar_sync(1, 32 * kBWarps);
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

PFN_cuTensorMapEncodeTiled_v12000 batch_encoder() {
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

bool bmap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t rows, uint64_t cols,
          uint32_t box_cols, uint32_t box_rows) {
  auto enc = batch_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_coop(const void *kern, int grid, int smem, cudaStream_t stream, void **args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

template <int NT>
cudaError_t proj_launch(const Launch &L, const ProjBatchParams &P, const BatchMaps &M, const CUtensorMap &tmUT,
                        int grid) {
  const int smem = kASmem + 1024;
  cudaError_t e;
  if ((e = ensure_dynamic_smem<k_lr_proj_batch<NT>>(smem)) != cudaSuccess) return e;
  k_lr_proj_batch<NT><<<grid, kBThreads, smem, L.stream>>>(P, M, tmUT, L.status);
  return cudaGetLastError();
}

template <int EPI, int F, int NPL, bool TOUT>
cudaError_t apply_launch(const Launch &L, const ApplyBatchParams &P, const BatchMaps &M, const CUtensorMap &tmU,
                         const CUtensorMap &tmPc, int grid) {
  const int smem = kBSmem + 1024;
  auto kern = k_lr_apply_batch<EPI, F, NPL, TOUT>;
  cudaError_t e;
  if ((e = ensure_dynamic_smem<k_lr_apply_batch<EPI, F, NPL, TOUT>>(smem)) != cudaSuccess) return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBThreads, smem)) != cudaSuccess) return e;
  if (per_sm < 1 || grid > per_sm * L.sms) return cudaErrorCooperativeLaunchTooLarge;
  int *status = L.status;
  void *args[] = {const_cast<ApplyBatchParams *>(&P), const_cast<BatchMaps *>(&M), const_cast<CUtensorMap *>(&tmU),
                  const_cast<CUtensorMap *>(&tmPc), &status};
  return launch_coop(reinterpret_cast<const void *>(kern), grid, smem, L.stream, args);
}

template <int NPL>
cudaError_t apply_dispatch(const Launch &L, int epi, int fmt, const ApplyBatchParams &P, const BatchMaps &M,
                           const CUtensorMap &tmU, const CUtensorMap &tmPc, int grid, bool t) {
  if (epi == LR_AMAX) return apply_launch<LR_AMAX, FMT_E4M3, NPL, false>(L, P, M, tmU, tmPc, grid);
  if (epi == LR_NVFP4)
    return t ? apply_launch<LR_NVFP4, FMT_E4M3, NPL, true>(L, P, M, tmU, tmPc, grid)
             : apply_launch<LR_NVFP4, FMT_E4M3, NPL, false>(L, P, M, tmU, tmPc, grid);
  if (fmt == GIFT_FMT_E5M2)
    return t ? apply_launch<LR_PACK_TENSOR, FMT_E5M2, NPL, true>(L, P, M, tmU, tmPc, grid)
             : apply_launch<LR_PACK_TENSOR, FMT_E5M2, NPL, false>(L, P, M, tmU, tmPc, grid);
  return t ? apply_launch<LR_PACK_TENSOR, FMT_E4M3, NPL, true>(L, P, M, tmU, tmPc, grid)
           : apply_launch<LR_PACK_TENSOR, FMT_E4M3, NPL, false>(L, P, M, tmU, tmPc, grid);
}

}  // namespace

// CTAs per row block: at most kBMaxTiles tiles each, the CTA's column range being its slice;
// one CTA per SM at most (pass B is cooperative).
int lr_batch_plan(int sms, int d_out, int d_in, int *cpr_out) {
  const int tiles_n = (d_in + kBN - 1) / kBN;
  const int tiles_m = (d_out + kBM - 1) / kBM;
  if (tiles_m > sms) return 0;
  int cpr = (tiles_n + kBMaxTiles - 1) / kBMaxTiles;
  const int spread = sms / tiles_m;
  if (spread > cpr) cpr = spread < tiles_n ? spread : tiles_n;
  if ((long long)cpr * tiles_m > sms) return 0;
  *cpr_out = cpr;
  return cpr * tiles_m;
}

size_t lr_batch_part_floats(int sms, int d_out, int d_in) {
  int cpr = 0;
  if (lr_batch_plan(sms, d_out, d_in, &cpr) <= 0) return 0;
  return (size_t)cpr * d_out * 32;
}

bool lr_encode_batch_ok(const Launch &L, const LrApply &a, int epi) {
  if (epi != LR_PACK_TENSOR && epi != LR_NVFP4 && epi != LR_AMAX) return false;
  if (a.inverse || !a.split || !a.grid_counter || !a.u_planes || !a.ut_planes) return false;
  if (!lr_apply_tc_ok(a, epi == LR_AMAX ? LR_PACK_TENSOR : epi) || !lr_proj_tc_ok(a.X, a.d_in, a.split) ||
      batch_encoder() == nullptr)
    return false;
  int cpr = 0;
  return lr_batch_plan(L.sms, a.d_out, a.d_in, &cpr) > 0;
}

// part: nb x lr_batch_part_floats floats; pc_planes: nb x 2 x d_out rows of 64 BF16.
// a.amax_ws[0..nb) zero for the tensors without a caller amax, a.grid_counter zero.
cudaError_t launch_lr_encode_batch(const Launch &L, int epi, int fmt, const LrApply &a, const float *mu,
                                   float *part, uint16_t *pc_planes, int nb, const LrEncodeItem *items) {
  if (nb < 1 || nb > kEncodeBatchMax) return cudaErrorInvalidValue;
  int cpr = 0;
  const int grid = lr_batch_plan(L.sms, a.d_out, a.d_in, &cpr);
  if (grid <= 0) return cudaErrorInvalidValue;
  const int NT = a.terms == 1 ? 2 : 3, NPL = NT - 1;
  BatchMaps M;
  std::memset(&M, 0, sizeof(M));
  bool tout = false;
  for (int k = 0; k < nb; ++k) {
    tout = tout || items[k].tout != nullptr;
    if (!bmap(&M.w[k], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, items[k].X, (uint64_t)a.d_out, (uint64_t)a.d_in, 32, kBM))
      return cudaErrorInvalidValue;
  }
  CUtensorMap tmUT, tmU, tmPc;
  if (!bmap(&tmUT, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.ut_planes, 96, (uint64_t)a.d_in, kBN, 32) ||
      !bmap(&tmU, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.u_planes, (uint64_t)NPL * a.d_in, 32, 32,
            kBGroupTiles * kBN) ||
      !bmap(&tmPc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, pc_planes, (uint64_t)nb * 2 * a.d_out, 32, 32, kBM))
    return cudaErrorInvalidValue;

  ProjBatchParams PA;
  PA.d_out = a.d_out;
  PA.d_in = a.d_in;
  PA.tiles_n = (a.d_in + kBN - 1) / kBN;
  PA.cpr = cpr;
  PA.nb = nb;
  PA.part = part;
  cudaError_t e = NT == 2 ? proj_launch<2>(L, PA, M, tmUT, grid) : proj_launch<3>(L, PA, M, tmUT, grid);
  if (e != cudaSuccess) return e;

  const long long items_r = (long long)nb * a.d_out * 16;
  const int rgrid = (int)((items_r + 255) / 256);
  if (NPL == 1)
    k_lr_pc_batch<1><<<rgrid, 256, 0, L.stream>>>(part, nb, cpr, a.d_out, mu, a.sigma, a.rank, pc_planes, L.status);
  else
    k_lr_pc_batch<2><<<rgrid, 256, 0, L.stream>>>(part, nb, cpr, a.d_out, mu, a.sigma, a.rank, pc_planes, L.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  ApplyBatchParams PB;
  std::memset(&PB, 0, sizeof(PB));
  PB.a = a;
  PB.tiles_n = PA.tiles_n;
  PB.cpr = cpr;
  PB.nb = nb;
  PB.reverse = 1;
  PB.grid_counter = a.grid_counter;
  for (int k = 0; k < nb; ++k) PB.item[k] = items[k];
  return NPL == 1 ? apply_dispatch<1>(L, epi, fmt, PB, M, tmU, tmPc, grid, tout)
                  : apply_dispatch<2>(L, epi, fmt, PB, M, tmU, tmPc, grid, tout);
}

}  // namespace gift
