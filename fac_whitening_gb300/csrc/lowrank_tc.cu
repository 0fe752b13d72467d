// Rank-r whitening apply on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17), with the sigma I
// completion: W~ = alpha W + (P diag(c)) U^T with P = W U (see lowrank.cu).  The rank-r
// product Pc U^T (K = 32) is a dense contraction over every element of the tile, so it runs
// on the tensor cores; the rest of the apply (alpha W, residual, amax, FP8/NVFP4 pack or
// FP32 store) is fused into the TMEM read-out.
//
// Tile: 128 rows x 64 columns per CTA, 128 threads.  D[128 x 64] (FP32, TMEM) =
// A[128 x 32] B[64 x 32]^T with A = Pc rows and B = U rows, both staged K-major in shared
// memory with the 128-byte swizzle (one 128-byte row per matrix row).  The W tile is
// prefetched with cp.async into padded shared memory while the operands are staged and the
// MMAs run; outputs (codes, FP32 values) are staged in shared memory and written back as
// coalesced row segments.  FP32 path: every
// operand is split exactly into three TF32 terms x = x1 + x2 + x3 and the six products with
// i + j <= 4 are accumulated (the dropped terms are below 2^-33 relative), which recovers
// FP32-level accuracy from TF32 MMAs (the split-precision idea of H. Ootomo and R. Yokota,
// "Recovering single precision accuracy from Tensor Cores while surpassing the FP32
// theoretical peak performance", IJHPCA 2022).  TC path: one TF32 product.
#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 64;
constexpr int kABytes = 128 * 128;               // Pc tile: 128 rows x 32 floats
constexpr int kBBytes = kTileN * 128;            // U tile: 64 rows x 32 floats
constexpr int kWStride = kTileN + 4;             // padded row (floats) of the staged W tile
constexpr int kWBytes = kTileM * kWStride * 4;
constexpr int kCStride = 80;                     // padded row (bytes) of the staged codes
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles for the MMA completion wait

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  const unsigned saddr = tc::smem_u32(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(valid ? 16 : 0));
}

// Split four values into TF32 terms and store them at the 128B-swizzled position of
// 16-byte chunk c of row r in `terms` operand copies `stride` bytes apart.
template <int TERMS>
__device__ __forceinline__ void put_split(uint8_t *base, int stride, int r, int c, float4 q) {
  const int off = r * 128 + ((c ^ (r & 7)) << 4);
  const float v[4] = {q.x, q.y, q.z, q.w};
  float t1[4], t2[4], t3[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    t1[e] = tc::tf32_round(v[e]);
    const float r1 = v[e] - t1[e];
    t2[e] = tc::tf32_round(r1);
    t3[e] = r1 - t2[e];
  }
  *reinterpret_cast<float4 *>(base + off) = make_float4(t1[0], t1[1], t1[2], t1[3]);
  if (TERMS > 1) {
    *reinterpret_cast<float4 *>(base + stride + off) = make_float4(t2[0], t2[1], t2[2], t2[3]);
    *reinterpret_cast<float4 *>(base + 2 * stride + off) = make_float4(t3[0], t3[1], t3[2], t3[3]);
  }
}

__device__ __forceinline__ float4 load_row4(const float *__restrict__ src, int ld, int gr, int nrows, int c,
                                            int kvalid) {
  float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
  if (gr < nrows) {
    const float *p = src + (size_t)gr * ld + 4 * c;
    if (ld == 32) {
      q = *reinterpret_cast<const float4 *>(p);
    } else {
      if (4 * c + 0 < kvalid) q.x = p[0];
      if (4 * c + 1 < kvalid) q.y = p[1];
      if (4 * c + 2 < kvalid) q.z = p[2];
      if (4 * c + 3 < kvalid) q.w = p[3];
    }
  }
  return q;
}

}  // namespace

// EPI: LR_AMAX, LR_PACK_TENSOR, LR_NVFP4, LR_STORE (see lowrank.cu).
template <int EPI, int F, int TERMS, bool TOUT>
__global__ void __launch_bounds__(128) k_lr_apply_tc(LrApply a, int *status) {
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = sm;                               // TERMS x Pc tile; reused for staged codes
  uint8_t *sB = sm + TERMS * kABytes;             // TERMS x U tile
  float *sW = reinterpret_cast<float *>(sB + TERMS * kBBytes);   // W tile, later the values
  __shared__ uint64_t mbar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[4];
  __shared__ int timed_out;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r0 = blockIdx.y * kTileM, c0 = blockIdx.x * kTileN;
  const int d_out = a.d_out, d_in = a.d_in;

  // 1. W tile -> shared memory (coalesced 16-byte pieces, zero outside the matrix)
#pragma unroll
  for (int i = 0; i < (kTileM * kTileN / 4) / 128; ++i) {
    const int q = i * 128 + tid;
    const int row = q >> 4, c = q & 15;
    const int gr = r0 + row, gc = c0 + 4 * c;
    const bool ok = gr < d_out && gc < d_in;
    cp_async16(sW + row * kWStride + 4 * c, ok ? (const void *)(a.X + (size_t)gr * d_in + gc) : (const void *)a.X, ok);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, kTileN);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&mbar, 1);
    tc::fence_mbar_init();
    timed_out = 0;
  }
  // 2. operands: all loads first, then split into TF32 terms and store swizzled
  {
    float4 qa[8], qb[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = i * 128 + tid;
      qa[i] = load_row4(a.Pc, 32, r0 + (q >> 3), d_out, q & 7, 32);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = i * 128 + tid;
      qb[i] = load_row4(a.U, a.rank, c0 + (q >> 3), d_in, q & 7, a.rank);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = i * 128 + tid;
      put_split<TERMS>(sA, kABytes, q >> 3, q & 7, qa[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = i * 128 + tid;
      put_split<TERMS>(sB, kBBytes, q >> 3, q & 7, qb[i]);
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  // 3. MMAs (one thread): D = sum of the TF32 term products
  if (tid == 0) {
    constexpr uint32_t idesc = tc::idesc_tf32(kTileM, kTileN);
    const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB);
    constexpr int np = (TERMS == 1) ? 1 : 6;
    const int pi[6] = {2, 1, 0, 1, 0, 0};
    const int pj[6] = {0, 1, 2, 0, 1, 0};
    uint32_t acc = 0;
#pragma unroll
    for (int p = 0; p < np; ++p) {
      const int ia = (TERMS == 1) ? 0 : pi[p], jb = (TERMS == 1) ? 0 : pj[p];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = tc::sdesc_kmajor_sw128(a0 + ia * kABytes + 32 * k);
        const uint64_t bd = tc::sdesc_kmajor_sw128(b0 + jb * kBBytes + 32 * k);
        tc::mma_tf32(tmem, ad, bd, idesc, acc);
        acc = 1;
      }
    }
    tc::mma_commit(&mbar);
  }

  // 4. wait for W and the accumulator
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  if (!tc::mbar_wait_bounded(&mbar, 0, kWaitBudget)) atomicExch(&timed_out, 1);
  tc::fence_after_sync();
  __syncthreads();
  if (timed_out) {
    if (tid == 0) set_status(status, GIFT_ERR_TIMEOUT);
    tc::mbar_wait_bounded(&mbar, 0, kWaitBudget);   // a second bounded chance before release
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, kTileN);
    }
    return;
  }

  // 5. epilogue: thread = tile row (TMEM lane); values alpha W + acc, written back in place
  const int lr = tid;
  const int row = r0 + lr;
  const bool row_ok = row < d_out;
  const double sg = (double)a.sigma[0];
  const float alpha = a.inverse ? (float)sqrt(sg) : (float)(1.0 / sqrt(sg));
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  float *wrow = sW + lr * kWStride;
  uint32_t m = 0;
#pragma unroll
  for (int cc = 0; cc < kTileN; cc += 32) {
    float v[32];
    tc::tmem_ld32(lane_addr + cc, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 w = *reinterpret_cast<const float4 *>(wrow + cc + 4 * q);
      const bool ok = row_ok && (c0 + cc + 4 * q) < d_in;
      float4 o;
      o.x = ok ? fmaf(alpha, w.x, v[4 * q + 0]) : 0.0f;
      o.y = ok ? fmaf(alpha, w.y, v[4 * q + 1]) : 0.0f;
      o.z = ok ? fmaf(alpha, w.z, v[4 * q + 2]) : 0.0f;
      o.w = ok ? fmaf(alpha, w.w, v[4 * q + 3]) : 0.0f;
      m = max(m, max(max(abs_bits(o.x), abs_bits(o.y)), max(abs_bits(o.z), abs_bits(o.w))));
      *reinterpret_cast<float4 *>(wrow + cc + 4 * q) = o;
    }
  }

  if (EPI == LR_AMAX) {
    m = warp_max_u32(m);
    if ((tid & 31) == 0) red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      m = max(max(red[0], red[1]), max(red[2], red[3]));
      atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws), m);
      if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    }
  } else if (EPI == LR_PACK_TENSOR) {
    const float amax = a.amax_in ? a.amax_in[0] : a.amax_ws[0];
    const ScalePair sp = scale_pair(amax, fmax_of<F>());
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
      if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      reinterpret_cast<float *>(a.scales)[0] = sp.s;
      if (a.amax_out) a.amax_out[0] = amax;
    }
    uint8_t *crow = sA + lr * kCStride;            // staged codes (operands are no longer read)
#pragma unroll
    for (int q = 0; q < kTileN / 16; ++q) {
      uint32_t c4[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float4 o = *reinterpret_cast<const float4 *>(wrow + 16 * q + 4 * h);
        c4[h] = pack4_fp8<F>(__fmul_rn(o.x, sp.m), __fmul_rn(o.y, sp.m), __fmul_rn(o.z, sp.m), __fmul_rn(o.w, sp.m));
      }
      *reinterpret_cast<uint4 *>(crow + 16 * q) = make_uint4(c4[0], c4[1], c4[2], c4[3]);
    }
    __syncthreads();
    // coalesced copy-out: 4 threads per 64-byte row segment
#pragma unroll
    for (int i = 0; i < (kTileM * kTileN / 16) / 128; ++i) {
      const int q = i * 128 + tid;
      const int rr = q >> 2, c = q & 3;
      const int gr = r0 + rr, gc = c0 + 16 * c;
      if (gr < d_out && gc < d_in)
        *reinterpret_cast<uint4 *>(a.codes + (size_t)gr * d_in + gc) = *reinterpret_cast<const uint4 *>(sA + rr * kCStride + 16 * c);
    }
  } else if (EPI == LR_NVFP4) {
    const float amax = a.amax_in ? a.amax_in[0] : a.amax_ws[0];
    const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
      if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      a.tscale[0] = s_t;
      if (a.amax_out) a.amax_out[0] = amax;
    }
    uint8_t *crow = sA + lr * kCStride;            // 32 code bytes, then 4 scale bytes
#pragma unroll
    for (int g = 0; g < kTileN / 16; ++g) {
      uint32_t gm = 0;
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) gm = max(gm, abs_bits(wrow[16 * g + i]));
      const Nv4Group grp = nvfp4_group(__uint_as_float(gm), s_t);
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(wrow[16 * g + i], grp.r);
      *reinterpret_cast<uint2 *>(crow + 8 * g) = make_uint2(pack8_e2m1(y), pack8_e2m1(y + 8));
      crow[32 + g] = grp.e_code;
    }
    __syncthreads();
    // codes: 32 bytes per row (2 threads x 16 bytes); scales: 4 bytes per row
#pragma unroll
    for (int i = 0; i < (kTileM * 2) / 128; ++i) {
      const int q = i * 128 + tid;
      const int rr = q >> 1, c = q & 1;
      const int gr = r0 + rr, gc = c0 + 32 * c;
      if (gr < d_out && gc < d_in)
        *reinterpret_cast<uint4 *>(a.codes + (((size_t)gr * d_in + gc) >> 1)) =
            *reinterpret_cast<const uint4 *>(sA + rr * kCStride + 16 * c);
    }
    {
      const int rr = tid, gr = r0 + rr;
      uint8_t *bscale = reinterpret_cast<uint8_t *>(a.scales);
      const uint8_t *sc = sA + rr * kCStride + 32;
      if (gr < d_out) {
#pragma unroll
        for (int g = 0; g < kTileN / 16; ++g)
          if (c0 + 16 * g < d_in) bscale[(size_t)gr * (d_in / kNvGroup) + (c0 + 16 * g) / kNvGroup] = sc[g];
      }
    }
  } else {   // LR_STORE
    __syncthreads();
  }

  // FP32 values out (decode output and/or the transformed copy): coalesced rows
  if (EPI == LR_STORE || TOUT) {
    if (EPI == LR_AMAX) __syncthreads();
    float *dst = (EPI == LR_STORE) ? a.out : a.tout;
#pragma unroll
    for (int i = 0; i < (kTileM * kTileN / 4) / 128; ++i) {
      const int q = i * 128 + tid;
      const int rr = q >> 4, c = q & 15;
      const int gr = r0 + rr, gc = c0 + 4 * c;
      if (gr < d_out && gc < d_in)
        *reinterpret_cast<float4 *>(dst + (size_t)gr * d_in + gc) = *reinterpret_cast<const float4 *>(sW + rr * kWStride + 4 * c);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTileN);
  }
}

// ---------------------------------------------------------------------------------------
size_t lr_apply_tc_smem(int terms) { return (size_t)terms * (kABytes + kBBytes) + kWBytes + 1024; }

// The tensor-core apply covers the per-tensor FP8, NVFP4, amax and store epilogues on the
// vectorised layout (d_in % 16 == 0, 16-byte aligned tensors, rank <= 32, no residual).
// Block scaling and error feedback use the FP32-SIMT apply in lowrank.cu.
bool lr_apply_tc_ok(const LrApply &a, int epi) {
  if (epi != LR_AMAX && epi != LR_PACK_TENSOR && epi != LR_NVFP4 && epi != LR_STORE) return false;
  bool ok = (a.d_in % 16 == 0) && aligned16(a.X) && aligned16(a.Pc) && !a.R && (!a.tout || aligned16(a.tout)) &&
            a.rank >= 1 && a.rank <= 32;
  if (a.rank == 32) ok = ok && aligned16(a.U);
  if (epi == LR_STORE) ok = ok && aligned16(a.out);
  if (epi == LR_PACK_TENSOR || epi == LR_NVFP4) ok = ok && aligned16(a.codes);
  if (epi == LR_NVFP4) ok = ok && (a.d_in % 32 == 0);   // 16-byte aligned rows of packed codes
  return ok;
}

template <int EPI, int F, int TERMS>
static cudaError_t tc_launch(const Launch &L, const LrApply &a) {
  const size_t smem = lr_apply_tc_smem(TERMS);
  dim3 grid((a.d_in + kTileN - 1) / kTileN, (a.d_out + kTileM - 1) / kTileM);
  cudaError_t e;
  if (a.tout) {
    if ((e = ensure_dynamic_smem<k_lr_apply_tc<EPI, F, TERMS, true>>((int)smem)) != cudaSuccess) return e;
    k_lr_apply_tc<EPI, F, TERMS, true><<<grid, 128, smem, L.stream>>>(a, L.status);
  } else {
    if ((e = ensure_dynamic_smem<k_lr_apply_tc<EPI, F, TERMS, false>>((int)smem)) != cudaSuccess) return e;
    k_lr_apply_tc<EPI, F, TERMS, false><<<grid, 128, smem, L.stream>>>(a, L.status);
  }
  return cudaGetLastError();
}

template <int TERMS>
static cudaError_t tc_dispatch(const Launch &L, int epi, int fmt, const LrApply &a) {
  switch (epi) {
    case LR_AMAX: return tc_launch<LR_AMAX, FMT_E4M3, TERMS>(L, a);
    case LR_STORE: return tc_launch<LR_STORE, FMT_E4M3, TERMS>(L, a);
    case LR_NVFP4: return tc_launch<LR_NVFP4, FMT_E4M3, TERMS>(L, a);
    case LR_PACK_TENSOR:
      return fmt == GIFT_FMT_E5M2 ? tc_launch<LR_PACK_TENSOR, FMT_E5M2, TERMS>(L, a)
                                  : tc_launch<LR_PACK_TENSOR, FMT_E4M3, TERMS>(L, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_lr_apply_tc(const Launch &L, int epi, int fmt, const LrApply &a, bool single_term) {
  return single_term ? tc_dispatch<1>(L, epi, fmt, a) : tc_dispatch<3>(L, epi, fmt, a);
}

}  // namespace gift
