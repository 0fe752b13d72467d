// K-FAC factor A = a^T a / T on the 5th-generation tensor cores (BF16 activations).
//
// GIFT reading notes (zhongzhuzhou.org), prerequisites, K-FAC eq. (4): the input-side factor
// is the second moment of the layer inputs over the batch.  a is T x d row-major BF16; the
// product is a dense contraction over T, so it runs on tcgen05 (kind::f16, FP32 accumulate
// in tensor memory).  Products of BF16 values are exact in FP32; the sum over T is the
// tensor core's FP32 accumulation (not round to nearest), which is why this kernel serves the
// TC precision of gift_factor_update and the FP32 precision keeps the SIMT path.
//
//   k_transpose_bf16  a (T x d) -> at (d x T), so that both operands are K-major rows.
//   k_syrk_tc         persistent over the lower 128 x 256 tiles of A (a tile is computed when
//                     some element has i >= j; the mirror kernel fills the upper triangle).
//                     Warp 8 streams the at rows of the tile (128 and 256 rows, 64 K per
//                     stage, 4 stages, TMA 128-byte swizzle); warp 9 issues 128 x 256 x 16
//                     MMAs into one of two 256-column TMEM accumulators; warps 0-7 read the
//                     finished accumulator (32 rows x 128 columns each), scale by 1/T and
//                     store 32 x 32 blocks through swizzled shared memory with TMA stores.
// Every mbarrier wait is clock-bounded and reports GIFT_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kSM = 128, kSN = 256, kSK = 64;
constexpr int kSStages = 4;
constexpr int kSWarps = 8;
constexpr int kSThreads = 32 * (kSWarps + 2);
constexpr int kSABytes = kSM * 128;          // 128 rows x 64 BF16
constexpr int kSBBytes = kSN * 128;          // 256 rows x 64 BF16
constexpr int kSStage = kSABytes + kSBBytes; // 48 KB
constexpr int kSOffStg = kSStages * kSStage; // epilogue staging: 8 warps x 4 KB
constexpr int kSSmem = kSOffStg + kSWarps * 4096;
constexpr long long kSWait = 4000000000LL;

struct SyrkParams {
  int d, T;
  float scale;
  int row_blocks, col_blocks, ntiles;
};

// lower-tile index -> (row block of 128, column block of 256)
__device__ __forceinline__ void tile_of(int t, int col_blocks, int &ti, int &tj) {
  int i = 0;
  for (;; ++i) {
    int cnt = i / 2 + 1;
    if (cnt > col_blocks) cnt = col_blocks;
    if (t < cnt) break;
    t -= cnt;
  }
  ti = i;
  tj = t;
}

__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(tmap),
               "r"(tc::smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

}  // namespace

// 64 x 64 tiles through shared memory; 16-byte loads and stores (d and T multiples of 64).
__global__ void __launch_bounds__(256) k_transpose_bf16(const uint16_t *__restrict__ x, int T, int d,
                                                        uint16_t *__restrict__ xt) {
  __shared__ uint16_t tile[64][64 + 8];
  const int i0 = blockIdx.x * 64, t0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 0; k < 2; ++k) {   // 64 rows x 8 chunks of 8 values
    const int q = k * 256 + tid, r = q >> 3, c = q & 7;
    const uint4 v = *reinterpret_cast<const uint4 *>(x + (size_t)(t0 + r) * d + i0 + 8 * c);
    const uint16_t *e = reinterpret_cast<const uint16_t *>(&v);
#pragma unroll
    for (int u = 0; u < 8; ++u) tile[8 * c + u][r] = e[u];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int q = k * 256 + tid, r = q >> 3, c = q & 7;
    uint4 v;
    uint16_t *e = reinterpret_cast<uint16_t *>(&v);
#pragma unroll
    for (int u = 0; u < 8; ++u) e[u] = tile[r][8 * c + u];
    *reinterpret_cast<uint4 *>(xt + (size_t)(i0 + r) * T + t0 + 8 * c) = v;
  }
}

__global__ void __launch_bounds__(kSThreads, 1) k_syrk_tc(const __grid_constant__ SyrkParams P,
                                                          const __grid_constant__ CUtensorMap tmA,
                                                          const __grid_constant__ CUtensorMap tmB,
                                                          const __grid_constant__ CUtensorMap tmC, int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[kSStages], empty[kSStages], afull[2], aempty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ksteps = P.T / kSK;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kSStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&afull[a], 1);
      tc::mbar_init(&aempty[a], kSWarps);
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
    if (!tc::mbar_wait_bounded(bar, parity, kSWait)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == kSWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      long long g = 0;   // stage uses so far
      int issued[kSStages] = {};
      bool ok = true;
      for (int t = blockIdx.x; t < P.ntiles && ok; t += gridDim.x) {
        int ti, tj;
        tile_of(t, P.col_blocks, ti, tj);
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = (int)(g % kSStages);
          if (!(ok = wait(&empty[s], (uint32_t)(((g / kSStages) & 1) ^ 1)))) break;
          uint8_t *st = sm + s * kSStage;
          tc::mbar_arrive_expect_tx(&full[s], kSStage);
          tc::tma_load_2d(st, &tmA, ks * kSK, ti * kSM, &full[s]);
          tc::tma_load_2d(st + kSABytes, &tmB, ks * kSK, tj * kSN, &full[s]);
          ++issued[s];
        }
      }
      if (failed) {
        for (int s = 0; s < kSStages; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&full[s], (uint32_t)((issued[s] - 1) & 1), kSWait);
      }
    }
  } else if (warp == kSWarps + 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kSM, kSN);
      long long g = 0;
      int n = 0;   // tiles of this CTA so far
      bool ok = true;
      for (int t = blockIdx.x; t < P.ntiles && ok; t += gridDim.x, ++n) {
        const int a = n & 1;
        if (!(ok = wait(&aempty[a], (uint32_t)(((n >> 1) & 1) ^ 1)))) break;
        tc::fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * kSN);
        for (int ks = 0; ks < ksteps; ++ks, ++g) {
          const int s = (int)(g % kSStages);
          if (!(ok = wait(&full[s], (uint32_t)((g / kSStages) & 1)))) break;
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sm + s * kSStage), b0 = a0 + kSABytes;
#pragma unroll
          for (int k = 0; k < kSK / 16; ++k)
            tc::mma_bf16(d, tc::sdesc_kmajor_sw128(a0 + 32 * k), tc::sdesc_kmajor_sw128(b0 + 32 * k), idesc,
                         (ks > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&afull[a]);
      }
    }
  } else {
    // ---------------- epilogue (warps 0-7): 32 rows x 128 columns each ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint8_t *stg = sm + kSOffStg + warp * 4096;
    int n = 0;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x, ++n) {
      int ti, tj;
      tile_of(t, P.col_blocks, ti, tj);
      const int a = n & 1;
      wait(&afull[a], (uint32_t)((n >> 1) & 1));
      tc::fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t raw[32];
        tc::tmem_ld32_nowait(tmem + lane_off + (uint32_t)(a * kSN + 128 * half + 32 * c), raw);
        tc::tmem_wait_ld(raw);
        if (lane == 0) bulk_wait_read0();   // the previous block has left the staging buffer
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4 *>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) =
              make_float4(__uint_as_float(raw[4 * q]) * P.scale, __uint_as_float(raw[4 * q + 1]) * P.scale,
                          __uint_as_float(raw[4 * q + 2]) * P.scale, __uint_as_float(raw[4 * q + 3]) * P.scale);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, stg, tj * kSN + 128 * half + 32 * c, ti * kSM + 32 * quarter);
          bulk_commit();
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&aempty[a]);
    }
    if (lane == 0) bulk_wait0();   // every store of this warp has completed
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

PFN_cuTensorMapEncodeTiled_v12000 syrk_encoder() {
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

bool smap(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *base, uint64_t rows, uint64_t cols,
          uint32_t box_cols, uint32_t box_rows) {
  auto enc = syrk_encoder();
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

bool syrk_tc_ok(int d, int T, const void *a, const void *at, const float *out) {
  return d % kSN == 0 && T % kSK == 0 && d >= kSN && aligned16(a) && aligned16(at) && aligned16(out) &&
         syrk_encoder() != nullptr;
}

size_t syrk_tc_scratch_bytes(int d, int T) { return (size_t)d * T * 2; }

cudaError_t launch_transpose_bf16(const Launch &L, const void *a, int T, int d, void *at) {
  k_transpose_bf16<<<dim3(d / 64, T / 64), 256, 0, L.stream>>>(static_cast<const uint16_t *>(a), T, d,
                                                                static_cast<uint16_t *>(at));
  return cudaGetLastError();
}

cudaError_t launch_syrk_tc(const Launch &L, const void *a, int T, int d, float scale, void *at, float *out) {
  k_transpose_bf16<<<dim3(d / 64, T / 64), 256, 0, L.stream>>>(static_cast<const uint16_t *>(a), T, d,
                                                                static_cast<uint16_t *>(at));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmA, tmB, tmC;
  if (!smap(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, at, (uint64_t)d, (uint64_t)T, kSK, kSM) ||
      !smap(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, at, (uint64_t)d, (uint64_t)T, kSK, kSN) ||
      !smap(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, out, (uint64_t)d, (uint64_t)d, 32, 32))
    return cudaErrorInvalidValue;
  SyrkParams P;
  P.d = d;
  P.T = T;
  P.scale = scale;
  P.row_blocks = d / kSM;
  P.col_blocks = d / kSN;
  int nt = 0;
  for (int i = 0; i < P.row_blocks; ++i) nt += (i / 2 + 1 < P.col_blocks) ? i / 2 + 1 : P.col_blocks;
  P.ntiles = nt;
  const int smem = kSSmem + 1024;
  if ((e = ensure_dynamic_smem<k_syrk_tc>(smem)) != cudaSuccess) return e;
  const int grid = nt < L.sms ? nt : L.sms;
  k_syrk_tc<<<grid, kSThreads, smem, L.stream>>>(P, tmA, tmB, tmC, L.status);
  return cudaGetLastError();
}

}  // namespace gift
