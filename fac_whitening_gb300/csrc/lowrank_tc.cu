// Rank-r whitening apply on the 5th-generation tensor cores: a persistent, warp-specialised
// pipeline (TMA loads -> tcgen05.mma into TMEM -> fused read-out).
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17), with the sigma I
// completion: W~ = alpha W + (P diag(c)) U^T with P = W U (see lowrank.cu).  The rank-r
// product Pc U^T (K = 32) is a dense contraction over every element of the tile, so it runs
// on the tensor cores; alpha W, the amax, the FP8/NVFP4 pack or the FP32 store are fused into
// the TMEM read-out.
//
// Tile: 128 rows x 64 columns.  D[128 x 64] (FP32, TMEM) = A[128 x 32] B[64 x 32]^T with
// A = rows of Pc and B = rows of U.  FP32 path: Pc and U are split exactly into three TF32
// terms (x = x1 + x2 + x3) beforehand and the six products with i + j <= 4 are accumulated,
// which recovers FP32-level accuracy from TF32 MMAs (the split-precision idea of H. Ootomo
// and R. Yokota, "Recovering single precision accuracy from Tensor Cores while surpassing the
// FP32 theoretical peak performance", IJHPCA 2022).  TC path: one TF32 product.
//
// One CTA per SM walks a contiguous range of tiles in row-block order (the A operand is
// loaded once per row block).  Warp 4 issues TMA loads (W tile as two 128 x 32 boxes, the B
// terms) into two stages; warp 5 issues the MMAs into two TMEM accumulators; warps 0-3 read
// out (one TMEM lane = one tile row per thread).  Full/empty mbarriers connect the roles;
// every wait is clock-bounded and reports GIFT_ERR_TIMEOUT instead of hanging.  The 128-byte
// TMA swizzle gives the tcgen05 K-major operand layout and conflict-free row reads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 64;
constexpr int kABytes = 128 * 128;            // 128 rows x 32 floats
constexpr int kBBytes = kTileN * 128;         // 64 rows x 32 floats
constexpr int kWBoxBytes = 128 * 128;         // 128 rows x 32 floats of W
constexpr long long kWaitBudget = 4000000000LL;

struct PipeParams {
  LrApply a;
  int tiles_n, tiles_total;
};

template <int TERMS>
struct Layout {
  static constexpr int a_off = 0;                                   // TERMS x A
  static constexpr int stage_bytes = 2 * kWBoxBytes + TERMS * kBBytes;
  static constexpr int stage_off = TERMS * kABytes;                 // 2 stages
  static constexpr int total = stage_off + 2 * stage_bytes;
};

__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

}  // namespace

template <int EPI, int F, int TERMS, bool TOUT>
__global__ void __launch_bounds__(192, 1) k_lr_apply_pipe(const __grid_constant__ PipeParams P,
                                                          const __grid_constant__ CUtensorMap tmW,
                                                          const __grid_constant__ CUtensorMap tmA,
                                                          const __grid_constant__ CUtensorMap tmB, int *status) {
  using Lay = Layout<TERMS>;
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_tfull[2], bar_tempty[2], bar_afull, bar_aempty, bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[4];
  __shared__ volatile int failed;

  const LrApply &a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = a.d_out, d_in = a.d_in;
  const int G = gridDim.x, b = blockIdx.x;
  const int t_begin = (int)(((long long)P.tiles_total * b) / G);
  const int t_end = (int)(((long long)P.tiles_total * (b + 1)) / G);

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 2 * kTileN);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], 4);
      tc::mbar_init(&bar_tfull[s], 1);
      tc::mbar_init(&bar_tempty[s], 4);
    }
    tc::mbar_init(&bar_afull, 1);
    tc::mbar_init(&bar_aempty, 1);
    tc::mbar_init(&bar_done, 1);
    tc::fence_mbar_init();
    failed = 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  auto wait = [&](uint64_t *bar, uint32_t parity) {
    if (failed) return false;
    if (!tc::mbar_wait_bounded(bar, parity, kWaitBudget)) {
      failed = 1;
      set_status(status, GIFT_ERR_TIMEOUT);
      return false;
    }
    return true;
  };

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int cur_rb = -1;
      uint32_t a_par = 0;
      int issued[2] = {0, 0}, a_issued = 0;
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int rb = t / P.tiles_n, cb = t - rb * P.tiles_n;
        const int s = i & 1;
        if (rb != cur_rb) {
          if (cur_rb >= 0) {
            if (!wait(&bar_aempty, a_par)) break;
            a_par ^= 1;
          }
          ++a_issued;
          tc::mbar_arrive_expect_tx(&bar_afull, TERMS * kABytes);
#pragma unroll
          for (int q = 0; q < TERMS; ++q)
            tc::tma_load_2d(sm + Lay::a_off + q * kABytes, &tmA, 0, q * d_out + rb * kTileM, &bar_afull);
          cur_rb = rb;
        }
        if (!wait(&bar_empty[s], ((i >> 1) & 1) ^ 1)) break;
        uint8_t *st = sm + Lay::stage_off + s * Lay::stage_bytes;
        tc::mbar_arrive_expect_tx(&bar_full[s], Lay::stage_bytes);
        tc::tma_load_2d(st, &tmW, cb * kTileN, rb * kTileM, &bar_full[s]);
        tc::tma_load_2d(st + kWBoxBytes, &tmW, cb * kTileN + 32, rb * kTileM, &bar_full[s]);
#pragma unroll
        for (int q = 0; q < TERMS; ++q)
          tc::tma_load_2d(st + 2 * kWBoxBytes + q * kBBytes, &tmB, 0, q * d_in + cb * kTileN, &bar_full[s]);
        ++issued[s];
      }
      if (failed) {
        // bounded drain of the loads still in flight before the CTA's shared memory goes away
        for (int s = 0; s < 2; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&bar_full[s], (uint32_t)((issued[s] - 1) & 1), kWaitBudget);
        if (a_issued) tc::mbar_wait_bounded(&bar_afull, (uint32_t)((a_issued - 1) & 1), kWaitBudget);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_tf32(kTileM, kTileN);
      int cur_rb = -1;
      uint32_t a_par = 0;
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int rb = t / P.tiles_n;
        const int s = i & 1;
        const uint32_t par = (i >> 1) & 1;
        if (rb != cur_rb) {
          if (!wait(&bar_afull, a_par)) break;
          a_par ^= 1;
          cur_rb = rb;
        }
        if (!wait(&bar_full[s], par)) break;
        if (!wait(&bar_tempty[s], par ^ 1)) break;
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(sm + Lay::a_off);
        const uint32_t b0 = tc::smem_u32(sm + Lay::stage_off + s * Lay::stage_bytes + 2 * kWBoxBytes);
        constexpr int np = (TERMS == 1) ? 1 : 6;
        const int pi[6] = {2, 1, 0, 1, 0, 0};
        const int pj[6] = {0, 1, 2, 0, 1, 0};
        uint32_t acc = 0;
#pragma unroll
        for (int p = 0; p < np; ++p) {
          const int ia = (TERMS == 1) ? 0 : pi[p], jb = (TERMS == 1) ? 0 : pj[p];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc::mma_tf32(tmem + s * kTileN, tc::sdesc_kmajor_sw128(a0 + ia * kABytes + 32 * k),
                         tc::sdesc_kmajor_sw128(b0 + jb * kBBytes + 32 * k), idesc, acc);
            acc = 1;
          }
        }
        tc::mma_commit(&bar_tfull[s]);
        const int nrb = (t + 1 < t_end) ? (t + 1) / P.tiles_n : -1;
        if (nrb != rb) tc::mma_commit(&bar_aempty);   // A of this row block may be replaced
      }
      // every MMA issued has landed in TMEM before the columns are freed
      tc::mma_commit(&bar_done);
      tc::mbar_wait_bounded(&bar_done, 0, kWaitBudget);
    }
  } else {
    // ---------------- read-out (warps 0-3): thread = tile row ----------------
    const double sg = (double)a.sigma[0];
    const float alpha = a.inverse ? (float)sqrt(sg) : (float)(1.0 / sqrt(sg));
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t m_run = 0;
    float amax = 0.0f, s_t = 0.0f;
    ScalePair sp = {0.0f, 0.0f};
    if (EPI == LR_PACK_TENSOR || EPI == LR_NVFP4) {
      amax = a.amax_in ? a.amax_in[0] : a.amax_ws[0];
      if (EPI == LR_PACK_TENSOR) sp = scale_pair(amax, fmax_of<F>());
      else s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
      if (b == 0 && tid == 0) {
        if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
        if (EPI == LR_PACK_TENSOR) reinterpret_cast<float *>(a.scales)[0] = sp.s;
        else a.tscale[0] = s_t;
        if (a.amax_out) a.amax_out[0] = amax;
      }
    }
    for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
      const int rb = t / P.tiles_n, cb = t - rb * P.tiles_n;
      const int s = i & 1;
      const uint32_t par = (i >> 1) & 1;
      const int r0 = rb * kTileM, c0 = cb * kTileN;
      // after a timeout the read-out still walks its tiles (on whatever the buffers hold, the
      // status already says the output is invalid) so that all four warps meet the same
      // named barriers; every later wait returns at once
      wait(&bar_tfull[s], par);
      wait(&bar_full[s], par);
      tc::fence_after_sync();
      float v[64];
      tc::tmem_ld32(lane_base + s * kTileN, v);
      tc::tmem_ld32(lane_base + s * kTileN + 32, v + 32);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_tempty[s]);

      uint8_t *st = sm + Lay::stage_off + s * Lay::stage_bytes;
      const int lr = tid;                      // tile row
      const int row = r0 + lr;
      // W (zero outside the matrix: TMA fill) -> values, written back in place when needed
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float4 *p = reinterpret_cast<float4 *>(st + h * kWBoxBytes + sw128(lr, c));
          const float4 w = *p;
          float *x = v + 32 * h + 4 * c;
          x[0] = fmaf(alpha, w.x, x[0]);
          x[1] = fmaf(alpha, w.y, x[1]);
          x[2] = fmaf(alpha, w.z, x[2]);
          x[3] = fmaf(alpha, w.w, x[3]);
          if (EPI == LR_STORE || TOUT) *p = make_float4(x[0], x[1], x[2], x[3]);
        }
      }
      if (EPI == LR_AMAX && row < d_out) {
        // term planes are stacked in one tensor, so rows / columns past the matrix edge hold
        // neighbouring data: they are kept out of the amax (and never stored)
#pragma unroll
        for (int e = 0; e < 64; e += 16)
          if (c0 + e < d_in) {
#pragma unroll
            for (int q = 0; q < 16; ++q) m_run = max(m_run, abs_bits(v[e + q]));
          }
      }
      if (EPI == LR_STORE || TOUT) {
        tc::named_bar_sync(1, 128);
        float *dst = (EPI == LR_STORE) ? a.out : a.tout;
#pragma unroll
        for (int k = 0; k < (kTileM * kTileN / 4) / 128; ++k) {
          const int q = k * 128 + tid;
          const int rr = q >> 4, c16 = q & 15;
          const int gr = r0 + rr, gc = c0 + 4 * c16;
          if (gr < d_out && gc < d_in)
            *reinterpret_cast<float4 *>(dst + (size_t)gr * d_in + gc) =
                *reinterpret_cast<const float4 *>(st + (c16 >> 3) * kWBoxBytes + sw128(rr, c16 & 7));
        }
        tc::named_bar_sync(1, 128);
      }
      if (EPI == LR_PACK_TENSOR) {
        // 64 codes per row -> the row's swizzled chunks 0..3 of box 0
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float *x = v + 16 * c + 4 * h;
            w4[h] = pack4_fp8<F>(__fmul_rn(x[0], sp.m), __fmul_rn(x[1], sp.m), __fmul_rn(x[2], sp.m),
                                 __fmul_rn(x[3], sp.m));
          }
          *reinterpret_cast<uint4 *>(st + sw128(lr, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        tc::named_bar_sync(1, 128);
#pragma unroll
        for (int k = 0; k < (kTileM * 4) / 128; ++k) {
          const int q = k * 128 + tid;
          const int rr = q >> 2, c = q & 3;
          const int gr = r0 + rr, gc = c0 + 16 * c;
          if (gr < d_out && gc < d_in)
            *reinterpret_cast<uint4 *>(a.codes + (size_t)gr * d_in + gc) = *reinterpret_cast<const uint4 *>(st + sw128(rr, c));
        }
        tc::named_bar_sync(1, 128);
      }
      if (EPI == LR_NVFP4) {
        uint8_t *bscale = reinterpret_cast<uint8_t *>(a.scales);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t gm = 0;
#pragma unroll
          for (int e = 0; e < 16; ++e) gm = max(gm, abs_bits(v[16 * g + e]));
          const Nv4Group grp = nvfp4_group(__uint_as_float(gm), s_t);
          float y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] = __fmul_rn(v[16 * g + e], grp.r);
          // the 8 code bytes of group g -> half of the row's swizzled chunk g / 2
          *reinterpret_cast<uint2 *>(st + sw128(lr, g >> 1) + 8 * (g & 1)) = make_uint2(pack8_e2m1(y), pack8_e2m1(y + 8));
          if (row < d_out && c0 + 16 * g < d_in)
            bscale[(size_t)row * (d_in / kNvGroup) + (c0 + 16 * g) / kNvGroup] = grp.e_code;
        }
        tc::named_bar_sync(1, 128);
#pragma unroll
        for (int k = 0; k < 2; ++k) {   // 128 rows x 2 chunks of 16 code bytes
          const int q = k * 128 + tid, rr = q >> 1, c = q & 1;
          const int gr = r0 + rr, gc = c0 + 32 * c;
          if (gr < d_out && gc < d_in)
            *reinterpret_cast<uint4 *>(a.codes + (((size_t)gr * d_in + gc) >> 1)) = *reinterpret_cast<const uint4 *>(st + sw128(rr, c));
        }
        tc::named_bar_sync(1, 128);
      }
      // this warp's generic-proxy writes into the stage are ordered before the TMA refill
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_empty[s]);
    }
    if (EPI == LR_AMAX) {
      m_run = warp_max_u32(m_run);
      if (lane == 0) red[warp] = m_run;
      tc::named_bar_sync(1, 128);
      if (tid == 0) {
        const uint32_t m = max(max(red[0], red[1]), max(red[2], red[3]));
        if (m) atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws), m);
        if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kTileN);
  }
}

// =========================================================================================
// exact TF32 split of a rows x ld matrix (first kvalid columns) into `terms` row-major
// rows x 32 planes, zero padded
// =========================================================================================
__global__ void k_split_terms(const float *__restrict__ src, int rows, int ld, int kvalid, int terms,
                              float *__restrict__ dst) {
  const size_t n = (size_t)rows * 32;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t r = i >> 5;
    const int k = (int)(i & 31);
    const float x = (k < kvalid) ? src[r * ld + k] : 0.0f;
    const float t1 = tc::tf32_round(x);
    const float r1 = x - t1;
    const float t2 = tc::tf32_round(r1);
    dst[i] = t1;
    if (terms > 1) {
      dst[n + i] = t2;
      dst[2 * n + i] = r1 - t2;
    }
  }
}

// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// FP32 row-major [rows][cols] tensor, box = 32 columns x box_rows rows, 128-byte swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t lr_pipe_split_floats(int d_out, int d_in) { return (size_t)3 * 32 * ((size_t)d_out + d_in); }

// The pipelined apply covers the per-tensor FP8, NVFP4, amax and store epilogues with
// d_in % 32 == 0 (TMA boxes of 32 columns, 16-byte aligned rows), 16-byte aligned tensors,
// rank <= 32, no residual and a split-term workspace; other cases use the FP32-SIMT apply
// in lowrank.cu.
bool lr_apply_tc_ok(const LrApply &a, int epi) {
  if (epi != LR_AMAX && epi != LR_PACK_TENSOR && epi != LR_NVFP4 && epi != LR_STORE) return false;
  if (!a.split) return false;
  bool ok = (a.d_in % 32 == 0) && aligned16(a.X) && aligned16(a.split) && !a.R &&
            (!a.tout || aligned16(a.tout)) && a.rank >= 1 && a.rank <= 32;
  if (epi == LR_STORE) ok = ok && aligned16(a.out);
  if (epi == LR_PACK_TENSOR || epi == LR_NVFP4) ok = ok && aligned16(a.codes);
  return ok && tensor_map_encoder() != nullptr;
}

// U terms go after the Pc terms (which the finalize writes) in the split workspace.
cudaError_t launch_lr_split_u(const Launch &L, const LrApply &a) {
  const int terms = (a.terms == 1) ? 1 : 3;
  float *uterms = a.split + (size_t)3 * 32 * a.d_out;
  const size_t n = (size_t)a.d_in * 32;
  int grid = (int)((n + 255) / 256);
  if (grid > L.sms * 8) grid = L.sms * 8;
  k_split_terms<<<grid, 256, 0, L.stream>>>(a.U, a.d_in, a.rank, a.rank, terms, uterms);
  return cudaGetLastError();
}

template <int EPI, int F, int TERMS>
static cudaError_t pipe_launch(const Launch &L, const LrApply &a) {
  CUtensorMap tmW, tmA, tmB;
  const float *pc = a.split;
  const float *ut = a.split + (size_t)3 * 32 * a.d_out;
  if (!make_map(&tmW, a.X, (uint64_t)a.d_out, (uint64_t)a.d_in, kTileM) ||
      !make_map(&tmA, pc, (uint64_t)TERMS * a.d_out, 32, kTileM) ||
      !make_map(&tmB, ut, (uint64_t)TERMS * a.d_in, 32, kTileN))
    return cudaErrorInvalidValue;
  PipeParams P;
  P.a = a;
  P.tiles_n = (a.d_in + kTileN - 1) / kTileN;
  const int tiles_m = (a.d_out + kTileM - 1) / kTileM;
  P.tiles_total = P.tiles_n * tiles_m;
  const int grid = P.tiles_total < L.sms ? P.tiles_total : L.sms;
  const int smem = Layout<TERMS>::total + 1024;
  cudaError_t e;
  if (a.tout) {
    if ((e = ensure_dynamic_smem<k_lr_apply_pipe<EPI, F, TERMS, true>>(smem)) != cudaSuccess) return e;
    k_lr_apply_pipe<EPI, F, TERMS, true><<<grid, 192, smem, L.stream>>>(P, tmW, tmA, tmB, L.status);
  } else {
    if ((e = ensure_dynamic_smem<k_lr_apply_pipe<EPI, F, TERMS, false>>(smem)) != cudaSuccess) return e;
    k_lr_apply_pipe<EPI, F, TERMS, false><<<grid, 192, smem, L.stream>>>(P, tmW, tmA, tmB, L.status);
  }
  return cudaGetLastError();
}

template <int TERMS>
static cudaError_t pipe_dispatch(const Launch &L, int epi, int fmt, const LrApply &a) {
  switch (epi) {
    case LR_AMAX: return pipe_launch<LR_AMAX, FMT_E4M3, TERMS>(L, a);
    case LR_STORE: return pipe_launch<LR_STORE, FMT_E4M3, TERMS>(L, a);
    case LR_NVFP4: return pipe_launch<LR_NVFP4, FMT_E4M3, TERMS>(L, a);
    case LR_PACK_TENSOR:
      return fmt == GIFT_FMT_E5M2 ? pipe_launch<LR_PACK_TENSOR, FMT_E5M2, TERMS>(L, a)
                                  : pipe_launch<LR_PACK_TENSOR, FMT_E4M3, TERMS>(L, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_lr_apply_tc(const Launch &L, int epi, int fmt, const LrApply &a, bool single_term) {
  return single_term ? pipe_dispatch<1>(L, epi, fmt, a) : pipe_dispatch<3>(L, epi, fmt, a);
}

}  // namespace gift
