// Rank-r input-side whitening of libgift (FP32 path).
//
// GIFT reading notes (zhongzhuzhou.org), simplification 1, eq. (16): W~ = W_g T_A with an
// input-side transform; simplification 2, eq. (17): A ~ U_r Lambda_r U_r^T with r = 32.
// Completing the rank-r factor with sigma I gives the invertible
//     T_A    = sigma^-1/2 I + U (diag(mu^-1/2) - sigma^-1/2) U^T
//     T_A^-1 = sigma^1/2  I + U (diag(mu^1/2)  - sigma^1/2)  U^T,
// so  W~ = sigma^-1/2 W + ((W U) diag(c)) U^T  and the map back (eq. (14)) has the same form.
//
// Three kernels:
//   k_lr_proj      P_s = X[:, J_s] U[J_s, :] for column slices J_s (split-K, FP32 partials);
//   k_lr_finalize  Pc = diag(c)-scaled sum of the slices, summed in FP64 in slice order;
//   k_lr_apply     V = alpha X + Pc U^T on a 2-D tile, fused with its consumer: amax, FP8
//                  pack (per tensor or per 128 x 128 block), NVFP4 pack, or FP32 store.
#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

// -------------------------------------------------------------------------------------
// projection: 128 rows x 32 outputs per CTA, 32-column chunks staged in shared memory.
// Threads: tz (2 halves of each chunk) x ty (16) x tx (8); rows ty + 16 i, outputs 4tx..4tx+3.
// -------------------------------------------------------------------------------------
constexpr int kProjRows = 128;
constexpr int kProjChunk = 32;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  const unsigned saddr = (unsigned)__cvta_generic_to_shared(smem);
  const int src = valid ? 16 : 0;   // 0 bytes read: the 16-byte destination is zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(src));
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
  const unsigned saddr = (unsigned)__cvta_generic_to_shared(smem);
  const int src = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(saddr), "l"(gmem), "r"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

template <bool VEC>
__global__ void __launch_bounds__(256, 2) k_lr_proj(const float *__restrict__ X, int d_out, int d_in,
                                                    const float *__restrict__ U, int rank,
                                                    float *__restrict__ part, int jspan) {
  // two stages of (X chunk, U chunk); stage buffers are reused for the final combine
  __shared__ __align__(16) float Xs[2][kProjRows][36];
  __shared__ __align__(16) float Us[2][kProjChunk][32];
  const int tid = threadIdx.x;
  const int tz = tid >> 7, t = tid & 127, tx = t & 7, ty = t >> 3;
  const int r0 = blockIdx.x * kProjRows;
  const int jbeg = blockIdx.y * jspan;
  const int jend = min(d_in, jbeg + jspan);
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[i][k] = 0.0f;

  // Stage chunk j0 into buffer b.  The vector path uses cp.async (16-byte X pieces,
  // 4-byte U elements, zero-filled outside the matrix); the scalar path plain loads.
  auto stage = [&](int b, int j0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = q * 256 + tid;
      const int row = idx >> 3, c4 = idx & 7;
      const int gr = r0 + row, gc = j0 + 4 * c4;
      if (VEC) {
        const bool ok = gr < d_out && gc < jend;
        cp_async16(&Xs[b][row][4 * c4], ok ? (const void *)(X + (size_t)gr * d_in + gc) : (const void *)X, ok);
      } else {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (gr < d_out) {
          const float *p = X + (size_t)gr * d_in;
          if (gc < jend) v.x = p[gc];
          if (gc + 1 < jend) v.y = p[gc + 1];
          if (gc + 2 < jend) v.z = p[gc + 2];
          if (gc + 3 < jend) v.w = p[gc + 3];
        }
        *reinterpret_cast<float4 *>(&Xs[b][row][4 * c4]) = v;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = q * 256 + tid;
      const int jj = idx >> 5, k = idx & 31;
      const int gj = j0 + jj;
      const bool ok = gj < jend && k < rank;
      if (VEC) cp_async4(&Us[b][jj][k], ok ? (const void *)(U + (size_t)gj * rank + k) : (const void *)U, ok);
      else Us[b][jj][k] = ok ? U[(size_t)gj * rank + k] : 0.0f;
    }
  };

  int b = 0;
  if (jbeg < jend) stage(0, jbeg);
  if (VEC) cp_async_commit();
  for (int j0 = jbeg; j0 < jend; j0 += kProjChunk) {
    const bool more = j0 + kProjChunk < jend;
    if (more) stage(b ^ 1, j0 + kProjChunk);
    if (VEC) {
      cp_async_commit();
      cp_async_wait<1>();   // the current stage has landed
    }
    __syncthreads();
#pragma unroll
    for (int jj = 0; jj < 16; jj += 4) {
      const int j = 16 * tz + jj;
      float4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = *reinterpret_cast<const float4 *>(&Xs[b][ty + 16 * i][j]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 bb = *reinterpret_cast<const float4 *>(&Us[b][j + q][4 * tx]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x = (q == 0) ? a[i].x : (q == 1) ? a[i].y : (q == 2) ? a[i].z : a[i].w;
          acc[i][0] = fmaf(x, bb.x, acc[i][0]);
          acc[i][1] = fmaf(x, bb.y, acc[i][1]);
          acc[i][2] = fmaf(x, bb.z, acc[i][2]);
          acc[i][3] = fmaf(x, bb.w, acc[i][3]);
        }
      }
    }
    __syncthreads();
    b ^= 1;
  }
  if (VEC) cp_async_wait<0>();
  __syncthreads();
  // combine the two chunk halves (tz) through shared memory, then write the slice partial
  float *red = &Xs[0][0][0];
  if (tz == 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4 *>(red + (ty + 16 * i) * 32 + 4 * tx) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  __syncthreads();
  if (tz == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = r0 + ty + 16 * i;
      if (row >= d_out) continue;
      const float4 o = *reinterpret_cast<const float4 *>(red + (ty + 16 * i) * 32 + 4 * tx);
      const float4 sum = make_float4(__fadd_rn(acc[i][0], o.x), __fadd_rn(acc[i][1], o.y),
                                     __fadd_rn(acc[i][2], o.z), __fadd_rn(acc[i][3], o.w));
      *reinterpret_cast<float4 *>(part + ((size_t)blockIdx.y * d_out + row) * 32 + 4 * tx) = sum;
    }
  }
}

// -------------------------------------------------------------------------------------
// finalize: Pc[row][k] = c_k * sum_s part[s][row][k]
//   whitening  c_k = mu_k^-1/2 - sigma^-1/2;  map back  c_k = mu_k^1/2 - sigma^1/2; 0 for k >= rank
// The 32 coefficients are formed once per CTA in FP64; the slice partials are added in
// slice order with a compensated (Kahan) FP32 sum, and the product is taken in FP64.
// -------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_lr_finalize(const float *__restrict__ part, int nsplit, int d_out,
                                                     const float *__restrict__ mu, const float *__restrict__ sigma,
                                                     int rank, bool inverse, float *__restrict__ Pc,
                                                     float *__restrict__ pc_terms, int terms, int *status) {
  __shared__ double coef[32];
  if (threadIdx.x < 32) {
    const int k = threadIdx.x;
    double c = 0.0;
    if (k < rank) {
      const double m = (double)mu[k], sg = (double)sigma[0];
      if (!(m > 0.0) || !(sg > 0.0)) {
        if (blockIdx.x == 0) set_status(status, GIFT_ERR_NOT_PD);
      } else {
        c = inverse ? (sqrt(m) - sqrt(sg)) : (1.0 / sqrt(m) - 1.0 / sqrt(sg));
      }
    }
    coef[k] = c;
  }
  __syncthreads();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= d_out * 32) return;
  float s = 0.0f, comp = 0.0f;
  for (int sp = 0; sp < nsplit; ++sp) {
    const float y = __fsub_rn(part[(size_t)sp * d_out * 32 + idx], comp);
    const float t = __fadd_rn(s, y);
    comp = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  const float pc = (float)(coef[idx & 31] * ((double)s - (double)comp));
  Pc[idx] = pc;
  if (pc_terms) {
    // BF16 term planes of Pc for the tensor-core apply (1 plane: TC path, 2: FP32 path)
    tc::write_term_planes(reinterpret_cast<uint16_t *>(pc_terms), (size_t)d_out, (size_t)(idx >> 5), idx & 31, pc,
                          terms == 1 ? 1 : 2);
  }
}

// -------------------------------------------------------------------------------------
// apply: tile (16 TM) rows x (64 NC) columns; thread (ty, tx) owns rows ty + 16 i and the
// 4-column chunks 4 tx + 64 n.  U^T is staged k-major with an XOR swizzle of the column
// (bits 2..4 by k / 4) so both the transposing stores and the float4 reads are free of
// bank conflicts.
// -------------------------------------------------------------------------------------
template <int EPI, int F, int TM, int NC, bool VEC, bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_lr_apply(LrApply a, int *status) {
  constexpr int BR = 16 * TM, BC = 64 * NC;
  __shared__ __align__(16) float Ps[BR][36];
  __shared__ __align__(16) float Us[32][BC];
  __shared__ uint32_t red[8];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int r0 = blockIdx.y * BR, c0 = blockIdx.x * BC;
  const int d_out = a.d_out, d_in = a.d_in, rank = a.rank;

  for (int idx = tid; idx < BR * 8; idx += 256) {
    const int row = idx >> 3, k4 = idx & 7;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + row < d_out) v = *reinterpret_cast<const float4 *>(a.Pc + (size_t)(r0 + row) * 32 + 4 * k4);
    *reinterpret_cast<float4 *>(&Ps[row][4 * k4]) = v;
  }
  for (int idx = tid; idx < BC * 8; idx += 256) {
    const int col = idx >> 3, k4 = idx & 7;
    const int gc = c0 + col;
    const int phys = col ^ (k4 << 2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 4 * k4 + e;
      Us[k][phys] = (gc < d_in && k < rank) ? a.U[(size_t)gc * rank + k] : 0.0f;
    }
  }
  __syncthreads();

  float acc[TM][NC][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int n = 0; n < NC; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.0f;

#pragma unroll
  for (int k = 0; k < 32; k += 4) {
    float4 pa[TM];
#pragma unroll
    for (int i = 0; i < TM; ++i) pa[i] = *reinterpret_cast<const float4 *>(&Ps[ty + 16 * i][k]);
    const int sw = (k >> 2) << 2;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        const float4 b = *reinterpret_cast<const float4 *>(&Us[k + kk][(4 * tx + 64 * n) ^ sw]);
#pragma unroll
        for (int i = 0; i < TM; ++i) {
          const float p = (kk == 0) ? pa[i].x : (kk == 1) ? pa[i].y : (kk == 2) ? pa[i].z : pa[i].w;
          acc[i][n][0] = fmaf(p, b.x, acc[i][n][0]);
          acc[i][n][1] = fmaf(p, b.y, acc[i][n][1]);
          acc[i][n][2] = fmaf(p, b.z, acc[i][n][2]);
          acc[i][n][3] = fmaf(p, b.w, acc[i][n][3]);
        }
      }
    }
  }

  // ---- V = alpha X + acc (+ R) -------------------------------------------------------
  const double sg = (double)a.sigma[0];
  const float alpha = a.inverse ? (float)sqrt(sg) : (float)(1.0 / sqrt(sg));
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = r0 + ty + 16 * i;
#pragma unroll
    for (int n = 0; n < NC; ++n) {
      const int col = c0 + 4 * tx + 64 * n;
      const size_t base = (size_t)row * d_in + col;
      float xv[4] = {0.f, 0.f, 0.f, 0.f}, rv[4] = {0.f, 0.f, 0.f, 0.f};
      if (row < d_out && col < d_in) {
        if (VEC) {
          const float4 x4 = *reinterpret_cast<const float4 *>(a.X + base);
          xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
          if (RES) {
            const float4 r4 = *reinterpret_cast<const float4 *>(a.R + base);
            rv[0] = r4.x; rv[1] = r4.y; rv[2] = r4.z; rv[3] = r4.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (col + e < d_in) {
              xv[e] = a.X[base + e];
              if (RES) rv[e] = a.R[base + e];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = fmaf(alpha, xv[e], acc[i][n][e]);
          if (RES) v = __fadd_rn(v, rv[e]);
          acc[i][n][e] = (VEC || col + e < d_in) ? v : 0.0f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) m = max(m, abs_bits(acc[i][n][e]));
    }
  }

  if (EPI == LR_STORE) {
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int row = r0 + ty + 16 * i;
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        const int col = c0 + 4 * tx + 64 * n;
        if (row >= d_out || col >= d_in) continue;
        const size_t base = (size_t)row * d_in + col;
        if (VEC) {
          *reinterpret_cast<float4 *>(a.out + base) =
              make_float4(acc[i][n][0], acc[i][n][1], acc[i][n][2], acc[i][n][3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (col + e < d_in) a.out[base + e] = acc[i][n][e];
        }
      }
    }
    return;
  }

  if (EPI == LR_AMAX || EPI == LR_BLOCK_AMAX) {
    m = block_max_u32<256>(m, red);
    if (tid == 0) {
      const int slot = (EPI == LR_BLOCK_AMAX) ? (blockIdx.y * gridDim.x + blockIdx.x) : 0;
      atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws) + slot, m);
      if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    }
    return;
  }

  // ---- scale ------------------------------------------------------------------------
  float amax;
  int tile = 0;
  if (EPI == LR_BLOCK) {
    m = block_max_u32<256>(m, red);
    tile = blockIdx.y * gridDim.x + blockIdx.x;
    amax = a.amax_in ? a.amax_in[tile] : __uint_as_float(m);
    if (tid == 0 && m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
  } else {
    amax = a.amax_in ? a.amax_in[0] : a.amax_ws[0];
  }

  if (EPI == LR_NVFP4) {
    const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
      if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      a.tscale[0] = s_t;
      if (a.amax_out) a.amax_out[0] = amax;
    }
    uint8_t *bscale = reinterpret_cast<uint8_t *>(a.scales);
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int row = r0 + ty + 16 * i;
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        const int col = c0 + 4 * tx + 64 * n;
        uint32_t gm = max(max(abs_bits(acc[i][n][0]), abs_bits(acc[i][n][1])),
                          max(abs_bits(acc[i][n][2]), abs_bits(acc[i][n][3])));
        gm = max(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 1));
        gm = max(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 2));
        if (row >= d_out || col >= d_in) continue;
        const Nv4Group g = nvfp4_group(__uint_as_float(gm), s_t);
        const size_t base = (size_t)row * d_in + col;
        const uint32_t c = pack4_e2m1(__fmul_rn(acc[i][n][0], g.r), __fmul_rn(acc[i][n][1], g.r),
                                      __fmul_rn(acc[i][n][2], g.r), __fmul_rn(acc[i][n][3], g.r));
        if (VEC) {
          *reinterpret_cast<uint16_t *>(a.codes + (base >> 1)) = (uint16_t)c;
        } else {
          a.codes[base >> 1] = (uint8_t)(c & 0xFF);
          a.codes[(base >> 1) + 1] = (uint8_t)((c >> 8) & 0xFF);
        }
        if ((tx & 3) == 0) bscale[(size_t)row * (d_in / kNvGroup) + col / kNvGroup] = g.e_code;
        if (TOUT) {
#pragma unroll
          for (int e = 0; e < 4; ++e) a.tout[base + e] = acc[i][n][e];
        }
        if (RES) {
          const float ev = dec_e4m3(g.e_code);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            a.R[base + e] = __fsub_rn(acc[i][n][e], nvfp4_deq((c >> (4 * e)) & 0xF, ev, s_t));
        }
      }
    }
    return;
  }

  // FP8 (per tensor or per block)
  const ScalePair sp = scale_pair(amax, fmax_of<F>());
  if (tid == 0) {
    if (EPI == LR_BLOCK) {
      reinterpret_cast<float *>(a.scales)[tile] = sp.s;
      if (a.amax_out) a.amax_out[tile] = amax;
    } else if (blockIdx.x == 0 && blockIdx.y == 0) {
      if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      reinterpret_cast<float *>(a.scales)[0] = sp.s;
      if (a.amax_out) a.amax_out[0] = amax;
    }
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int row = r0 + ty + 16 * i;
#pragma unroll
    for (int n = 0; n < NC; ++n) {
      const int col = c0 + 4 * tx + 64 * n;
      if (row >= d_out || col >= d_in) continue;
      const size_t base = (size_t)row * d_in + col;
      const uint32_t c = pack4_fp8<F>(__fmul_rn(acc[i][n][0], sp.m), __fmul_rn(acc[i][n][1], sp.m),
                                      __fmul_rn(acc[i][n][2], sp.m), __fmul_rn(acc[i][n][3], sp.m));
      float e4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        e4[e] = RES ? __fsub_rn(acc[i][n][e], __fmul_rn(dec_fp8<F>((c >> (8 * e)) & 0xFF), sp.s)) : 0.0f;
      if (VEC) {
        *reinterpret_cast<uint32_t *>(a.codes + base) = c;
        if (TOUT) *reinterpret_cast<float4 *>(a.tout + base) = make_float4(acc[i][n][0], acc[i][n][1], acc[i][n][2], acc[i][n][3]);
        if (RES) *reinterpret_cast<float4 *>(a.R + base) = make_float4(e4[0], e4[1], e4[2], e4[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (col + e >= d_in) continue;
          a.codes[base + e] = (uint8_t)((c >> (8 * e)) & 0xFF);
          if (TOUT) a.tout[base + e] = acc[i][n][e];
          if (RES) a.R[base + e] = e4[e];
        }
      }
    }
  }
}

// -------------------------------------------------------------------------------------
// launchers
// -------------------------------------------------------------------------------------
int lr_proj_splits(int sms, int d_out, int d_in) {
  const int rowblocks = (d_out + kProjRows - 1) / kProjRows;
  const int chunks = (d_in + kProjChunk - 1) / kProjChunk;
  int want = (2 * sms + rowblocks - 1) / rowblocks;   // about two CTAs per SM
  if (want < 1) want = 1;
  if (want > chunks) want = chunks;
  const int per = (chunks + want - 1) / want;          // chunks per slice
  return (chunks + per - 1) / per;
}

cudaError_t launch_lr_proj(const Launch &L, const float *X, int d_out, int d_in, const float *U, int rank,
                           float *part, int nsplit) {
  const int chunks = (d_in + kProjChunk - 1) / kProjChunk;
  const int per = (chunks + nsplit - 1) / nsplit;
  const int jspan = per * kProjChunk;
  dim3 grid((d_out + kProjRows - 1) / kProjRows, nsplit);
  const bool vec = (d_in % 4 == 0) && aligned16(X) && (((uintptr_t)U & 3u) == 0);
  if (vec) k_lr_proj<true><<<grid, 256, 0, L.stream>>>(X, d_out, d_in, U, rank, part, jspan);
  else k_lr_proj<false><<<grid, 256, 0, L.stream>>>(X, d_out, d_in, U, rank, part, jspan);
  return cudaGetLastError();
}

cudaError_t lr_prepare_all(const Launch &L, const float *U, const float *mu, const float *sigma, int rank,
                           const float *X, int d_out, int d_in, bool inverse, bool tc_precision, float *part,
                           float *Pc, float *split, const void *cached_planes) {
  cudaError_t e;
  if (split && lr_proj_tc_ok(X, d_in, split)) {
    const uint16_t *u = nullptr, *ut = nullptr;
    lr_u_planes(cached_planes, split, d_out, d_in, &u, &ut);
    if (!cached_planes) {
      if ((e = launch_lr_split_u_all(L, U, d_out, d_in, rank, tc_precision ? 1 : 2, split)) != cudaSuccess) return e;
    } else {
      const LrPlanes pl = lr_planes(split, d_out, d_in);   // the projection's barrier word
      if ((e = cudaMemsetAsync(pl.counters, 0, sizeof(unsigned int), L.stream)) != cudaSuccess) return e;
    }
    return launch_lr_proj_tc(L, X, d_out, d_in, mu, sigma, rank, inverse, tc_precision, part, Pc, split, ut);
  }
  const int nsplit = lr_proj_splits(L.sms, d_out, d_in);
  if ((e = launch_lr_proj(L, X, d_out, d_in, U, rank, part, nsplit)) != cudaSuccess) return e;
  float *pc_terms = (split && d_in % 32 == 0) ? split : nullptr;
  const int terms = tc_precision ? 1 : 3;
  if ((e = launch_lr_finalize(L, part, nsplit, d_out, mu, sigma, rank, inverse, Pc, pc_terms, terms)) != cudaSuccess)
    return e;
  if (!pc_terms || cached_planes) return cudaSuccess;
  LrApply a{};
  a.U = U;
  a.rank = rank;
  a.d_out = d_out;
  a.d_in = d_in;
  a.terms = terms;
  a.split = split;
  return launch_lr_split_u(L, a);
}

size_t lr_part_floats(int sms, int d_out, int d_in) {
  int ns = lr_proj_splits(sms, d_out, d_in);
  const int nt = lr_proj_tc_splits(sms, d_out, d_in);
  if (nt > ns) ns = nt;
  return (size_t)ns * d_out * 32;
}

cudaError_t launch_lr_finalize(const Launch &L, const float *part, int nsplit, int d_out, const float *mu,
                               const float *sigma, int rank, bool inverse, float *Pc, float *pc_terms, int terms) {
  const int n = d_out * 32;
  k_lr_finalize<<<(n + 255) / 256, 256, 0, L.stream>>>(part, nsplit, d_out, mu, sigma, rank, inverse, Pc, pc_terms,
                                                       terms, L.status);
  return cudaGetLastError();
}

template <int EPI, int F, int TM, int NC>
static void apply_dispatch(const Launch &L, const LrApply &a, bool vec) {
  dim3 grid((a.d_in + 64 * NC - 1) / (64 * NC), (a.d_out + 16 * TM - 1) / (16 * TM));
  const bool res = a.R != nullptr, to = a.tout != nullptr;
#define LRA(V, RS, TO) k_lr_apply<EPI, F, TM, NC, V, RS, TO><<<grid, 256, 0, L.stream>>>(a, L.status)
  if (vec) {
    if (res) { if (to) LRA(true, true, true); else LRA(true, true, false); }
    else { if (to) LRA(true, false, true); else LRA(true, false, false); }
  } else {
    if (res) { if (to) LRA(false, true, true); else LRA(false, true, false); }
    else { if (to) LRA(false, false, true); else LRA(false, false, false); }
  }
#undef LRA
}

cudaError_t launch_lr_apply(const Launch &L, int epi, int fmt, const LrApply &a) {
  if (lr_apply_tc_ok(a, epi)) return launch_lr_apply_tc(L, epi, fmt, a, a.terms == 1);
  bool vec = (a.d_in % 4 == 0) && aligned16(a.X) && (!a.R || aligned16(a.R)) && (!a.tout || aligned16(a.tout));
  if (epi == LR_STORE) vec = vec && aligned16(a.out);
  if (epi == LR_PACK_TENSOR || epi == LR_BLOCK) vec = vec && (((uintptr_t)a.codes & 3u) == 0);
  if (epi == LR_NVFP4) vec = vec && (((uintptr_t)a.codes & 1u) == 0);
  const bool e5 = (fmt == GIFT_FMT_E5M2);
  switch (epi) {
    case LR_AMAX: apply_dispatch<LR_AMAX, FMT_E4M3, 4, 4>(L, a, vec); break;
    case LR_BLOCK_AMAX: apply_dispatch<LR_BLOCK_AMAX, FMT_E4M3, 8, 2>(L, a, vec); break;
    case LR_STORE: apply_dispatch<LR_STORE, FMT_E4M3, 4, 4>(L, a, vec); break;
    case LR_NVFP4: apply_dispatch<LR_NVFP4, FMT_E4M3, 4, 4>(L, a, vec); break;
    case LR_PACK_TENSOR:
      if (e5) apply_dispatch<LR_PACK_TENSOR, FMT_E5M2, 4, 4>(L, a, vec);
      else apply_dispatch<LR_PACK_TENSOR, FMT_E4M3, 4, 4>(L, a, vec);
      break;
    case LR_BLOCK:
      if (e5) apply_dispatch<LR_BLOCK, FMT_E5M2, 8, 2>(L, a, vec);
      else apply_dispatch<LR_BLOCK, FMT_E4M3, 8, 2>(L, a, vec);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gift
