// Streaming quantisation kernels of libgift: amax, FP8 / NVFP4 pack with optional error
// feedback, replica dequantise-and-average, boundary-hit counting.
//
// GIFT reading notes (zhongzhuzhou.org):
//   prerequisites, "What FP8 is" .. s = amax(X)/FP8_MAX per tensor or per block, quantise;
//   Algorithm 1 ...................... Scale, AllReduceMax, Q, AllReduceSum, Dequantize / N,
//                                      error feedback U~ = U + R, R <- U~ - Dequantize(Q(U~));
//   simplification 3 ................. count codes on the upper / lower FP8 boundary.
// GIFT abstract (shd-paper.top): NVFP4 as the second low-precision format.
//
// Every kernel is HBM-bound: 16-byte loads and stores, grid-stride loops sized to the SM
// count, warp-shuffle reductions and one atomic per CTA (or warp).  The shared-scale encode of
// several replicas is one cooperative launch with one grid-wide barrier between its amax and
// pack passes.
#include <cstring>

#include "kernels.cuh"

namespace gift {

__device__ __forceinline__ float4 add4(float4 v, float4 q) {
  return make_float4(__fadd_rn(v.x, q.x), __fadd_rn(v.y, q.y), __fadd_rn(v.z, q.z), __fadd_rn(v.w, q.w));
}

// =====================================================================================
// amax of x (+ r): max of |value| bit patterns; non-finite values compare above every
// finite one, so a result >= 0x7F800000 flags NaN/Inf.
// =====================================================================================
template <bool VEC, bool RES>
__global__ void __launch_bounds__(256) k_amax(const float *__restrict__ x, const float *__restrict__ r,
                                              size_t n, uint32_t *__restrict__ amax_bits, int *status) {
  __shared__ uint32_t red[8];
  uint32_t m = 0;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t done = 0;
  if (VEC) {
    const size_t n4 = n >> 2;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const float4 *r4 = reinterpret_cast<const float4 *>(r);
    for (size_t i = tid; i < n4; i += stride) {
      float4 v = x4[i];
      if (RES) v = add4(v, r4[i]);
      m = max(m, max(max(abs_bits(v.x), abs_bits(v.y)), max(abs_bits(v.z), abs_bits(v.w))));
    }
    done = n4 << 2;
  }
  for (size_t i = done + tid; i < n; i += stride) {
    float v = x[i];
    if (RES) v = __fadd_rn(v, r[i]);
    m = max(m, abs_bits(v));
  }
  m = block_max_u32<256>(m, red);
  if (threadIdx.x == 0) {
    if (m) atomicMax(amax_bits, m);
    if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
  }
}

// =====================================================================================
// per-tensor FP8 pack: code = RNE_sat(fl(v * m)), v = x (+ r); optional residual update
// r <- v - fl(value(code) * s) and transformed copy.
// =====================================================================================
template <int F, bool VEC, bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_pack_tensor(const float *__restrict__ x, float *__restrict__ r,
                                                     size_t n, const float *__restrict__ amax_ptr,
                                                     uint8_t *__restrict__ codes, float *__restrict__ scale_out,
                                                     float *__restrict__ amax_out, float *__restrict__ tout,
                                                     int *status) {
  const float amax = *amax_ptr;
  const ScalePair sp = scale_pair(amax, fmax_of<F>());
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
    scale_out[0] = sp.s;
    if (amax_out) amax_out[0] = amax;
  }
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t done = 0;
  if (VEC) {
    const size_t n4 = n >> 2;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    float4 *r4 = reinterpret_cast<float4 *>(r);
    float4 *t4 = reinterpret_cast<float4 *>(tout);
    uint32_t *c4 = reinterpret_cast<uint32_t *>(codes);
    for (size_t i = tid; i < n4; i += stride) {
      float4 v = x4[i];
      if (RES) v = add4(v, r4[i]);
      if (TOUT) t4[i] = v;
      const uint32_t c = pack4_fp8<F>(__fmul_rn(v.x, sp.m), __fmul_rn(v.y, sp.m), __fmul_rn(v.z, sp.m),
                                      __fmul_rn(v.w, sp.m));
      c4[i] = c;
      if (RES) {
        float4 e;
        e.x = __fsub_rn(v.x, __fmul_rn(dec_fp8<F>(c & 0xFF), sp.s));
        e.y = __fsub_rn(v.y, __fmul_rn(dec_fp8<F>((c >> 8) & 0xFF), sp.s));
        e.z = __fsub_rn(v.z, __fmul_rn(dec_fp8<F>((c >> 16) & 0xFF), sp.s));
        e.w = __fsub_rn(v.w, __fmul_rn(dec_fp8<F>(c >> 24), sp.s));
        r4[i] = e;
      }
    }
    done = n4 << 2;
  }
  for (size_t i = done + tid; i < n; i += stride) {
    float v = x[i];
    if (RES) v = __fadd_rn(v, r[i]);
    if (TOUT) tout[i] = v;
    const uint8_t c = pack1_fp8<F>(__fmul_rn(v, sp.m));
    codes[i] = c;
    if (RES) r[i] = __fsub_rn(v, __fmul_rn(dec_fp8<F>(c), sp.s));
  }
}

// =====================================================================================
// The same amax and pack over several tensors of one size in one launch (the replicas of a
// layer): the CTAs walk the tensors in order, each thread with four 16-byte loads in flight.
// Per element the arithmetic is that of k_amax / k_pack_tensor.
// =====================================================================================
// max |x| bit pattern over the thread's grid-stride share of n4 float4s
__device__ __forceinline__ uint32_t amax_pass(const float4 *__restrict__ x4, size_t n4, size_t tid, size_t stride) {
  uint32_t m = 0;
  size_t i = tid;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = x4[i + u * stride];   // kept in L2 for the pack pass
#pragma unroll
    for (int u = 0; u < 4; ++u)
      m = max(m, max(max(abs_bits(v[u].x), abs_bits(v[u].y)), max(abs_bits(v[u].z), abs_bits(v[u].w))));
  }
  for (; i < n4; i += stride) {
    const float4 v = x4[i];
    m = max(m, max(max(abs_bits(v.x), abs_bits(v.y)), max(abs_bits(v.z), abs_bits(v.w))));
  }
  return m;
}

// codes of the thread's grid-stride share of n4 float4s with multiplier sp.m; inputs and codes
// are marked evict-first in L2 (neither is read again by this launch)
template <int F>
__device__ __forceinline__ void pack_pass(const float4 *__restrict__ x4, uint32_t *__restrict__ c4, size_t n4,
                                          size_t tid, size_t stride, const ScalePair sp) {
  auto code = [&](const float4 &v) {
    return pack4_fp8<F>(__fmul_rn(v.x, sp.m), __fmul_rn(v.y, sp.m), __fmul_rn(v.z, sp.m), __fmul_rn(v.w, sp.m));
  };
  size_t i = tid;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(x4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(c4 + i + u * stride, code(v[u]));
  }
  for (; i < n4; i += stride) __stcs(c4 + i, code(__ldcs(x4 + i)));
}

// the same two passes over two tensors at once (eight 16-byte loads in flight per thread)
__device__ __forceinline__ uint32_t amax_pass2(const float4 *__restrict__ xa, const float4 *__restrict__ xb, size_t n4,
                                               size_t tid, size_t stride) {
  uint32_t m = 0;
  size_t i = tid;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = xa[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[4 + u] = xb[i + u * stride];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      m = max(m, max(max(abs_bits(v[u].x), abs_bits(v[u].y)), max(abs_bits(v[u].z), abs_bits(v[u].w))));
  }
  for (; i < n4; i += stride) {
    const float4 v = xa[i], w = xb[i];
    m = max(m, max(max(abs_bits(v.x), abs_bits(v.y)), max(abs_bits(v.z), abs_bits(v.w))));
    m = max(m, max(max(abs_bits(w.x), abs_bits(w.y)), max(abs_bits(w.z), abs_bits(w.w))));
  }
  return m;
}

template <int F>
__device__ __forceinline__ void pack_pass2(const float4 *__restrict__ xa, uint32_t *__restrict__ ca,
                                           const float4 *__restrict__ xb, uint32_t *__restrict__ cb, size_t n4,
                                           size_t tid, size_t stride, const ScalePair sp) {
  auto code = [&](const float4 &v) {
    return pack4_fp8<F>(__fmul_rn(v.x, sp.m), __fmul_rn(v.y, sp.m), __fmul_rn(v.z, sp.m), __fmul_rn(v.w, sp.m));
  };
  size_t i = tid;
  for (; i + 3 * stride < n4; i += 4 * stride) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(xa + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) v[4 + u] = __ldcs(xb + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(ca + i + u * stride, code(v[u]));
#pragma unroll
    for (int u = 0; u < 4; ++u) __stcs(cb + i + u * stride, code(v[4 + u]));
  }
  for (; i < n4; i += stride) {
    __stcs(ca + i, code(__ldcs(xa + i)));
    __stcs(cb + i, code(__ldcs(xb + i)));
  }
}

__global__ void __launch_bounds__(256) k_amax_multi(MultiArgs a, int R, size_t n4, int *status) {
  __shared__ uint32_t red[8];
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int t = 0; t < R; ++t) {
    uint32_t m = amax_pass(reinterpret_cast<const float4 *>(a.x[t]), n4, tid, stride);
    m = block_max_u32<256>(m, red);
    if (threadIdx.x == 0) {
      if (m) atomicMax(a.amax_bits[t], m);
      if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    }
  }
}

template <int F>
__global__ void __launch_bounds__(256) k_pack_tensor_multi(MultiArgs a, int R, size_t n4, int *status) {
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int t = 0; t < R; ++t) {
    const float amax = *a.amax_in[t];
    const ScalePair sp = scale_pair(amax, fmax_of<F>());
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      a.scale[t][0] = sp.s;
      if (a.amax_out[t]) a.amax_out[t][0] = amax;
    }
    pack_pass<F>(reinterpret_cast<const float4 *>(a.x[t]), reinterpret_cast<uint32_t *>(a.codes[t]), n4, tid,
                 stride, sp);
  }
}

// =====================================================================================
// Boundary hits of several tensors of any sizes (the profiler over a model's layers): one
// launch takes every tensor's amax, one launch counts every tensor's hits with its own scale,
// the tensors taken last to first so that the count reads first what the amax pass read last.
// Per tensor the arithmetic is that of k_amax + k_hits_tensor.
// =====================================================================================
__global__ void __launch_bounds__(256) k_amax_multi_var(HitsArgs a, int T, uint32_t *amax_bits, int *status) {
  __shared__ uint32_t red[8];
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int t = 0; t < T; ++t) {
    const float *x = a.x[t];
    const size_t n = a.n[t];
    uint32_t m = 0;
    size_t done = 0;
    if ((((uintptr_t)x) & 15u) == 0) {
      m = amax_pass(reinterpret_cast<const float4 *>(x), n >> 2, tid, stride);
      done = (n >> 2) << 2;
    }
    for (size_t i = done + tid; i < n; i += stride) m = max(m, abs_bits(x[i]));
    m = block_max_u32<256>(m, red);
    if (threadIdx.x == 0) {
      if (m) atomicMax(amax_bits + t, m);
      if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    }
  }
}

template <int F>
__global__ void __launch_bounds__(256) k_hits_multi_var(HitsArgs a, int T, const uint32_t *__restrict__ amax_bits,
                                                        unsigned long long *__restrict__ counts) {
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int t = T - 1; t >= 0; --t) {
    const float *x = a.x[t];
    const size_t n = a.n[t];
    const ScalePair sp = scale_pair(__uint_as_float(amax_bits[t]), fmax_of<F>());
    uint32_t up = 0, lo = 0;
    auto tally4 = [&](const float4 &v) {
      const uint32_t c = pack4_fp8<F>(__fmul_rn(v.x, sp.m), __fmul_rn(v.y, sp.m), __fmul_rn(v.z, sp.m),
                                      __fmul_rn(v.w, sp.m));
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t mag = (c >> (8 * e)) & 0x7Fu;
        up += (mag == maxcode_of<F>());
        lo += (mag == 0u && vv[e] != 0.0f);
      }
    };
    size_t done = 0;
    if ((((uintptr_t)x) & 15u) == 0) {
      const float4 *x4 = reinterpret_cast<const float4 *>(x);
      const size_t n4 = n >> 2;
      size_t i = tid;
      for (; i + 7 * stride < n4; i += 8 * stride) {   // eight loads in flight
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldcs(x4 + i + u * stride);
#pragma unroll
        for (int u = 0; u < 8; ++u) tally4(v[u]);
      }
      for (; i < n4; i += stride) tally4(__ldcs(x4 + i));
      done = n4 << 2;
    }
    for (size_t i = done + tid; i < n; i += stride) {
      const float v = x[i];
      const uint32_t mag = pack1_fp8<F>(__fmul_rn(v, sp.m)) & 0x7Fu;
      up += (mag == maxcode_of<F>());
      lo += (mag == 0u && v != 0.0f);
    }
    up = warp_add_u32(up);
    lo = warp_add_u32(lo);
    if ((threadIdx.x & 31) == 0) {
      if (up) atomicAdd(counts + 3 * (size_t)t + 0, (unsigned long long)up);
      if (lo) atomicAdd(counts + 3 * (size_t)t + 1, (unsigned long long)lo);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(counts + 3 * (size_t)t + 2, (unsigned long long)n);
  }
}

// =====================================================================================
// The replicas of one tensor encoded with one shared scale (the synchronised scale of the
// Euclidean path: the max over the replicas of their amax) in one cooperative launch: the
// amax pass over every replica, a grid-wide barrier, then the pack of every replica with the
// shared amax, last replica first, so that the pack reads first what the amax pass read
// last and L2 still holds.  Per element the arithmetic is that of the two launches
// k_amax_multi + k_pack_tensor_multi.  ws[0] (amax bit pattern) and ws[1] (barrier count)
// are zero on entry.  The barrier wait is bounded: a CTA that gives up sets
// GIFT_ERR_TIMEOUT and writes no codes.
// =====================================================================================
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <int F>
__global__ void __launch_bounds__(256) k_encode_shared(MultiArgs a, int R, size_t n4, uint32_t *ws,
                                                       float *shared_out, long long wait_budget, int *status) {
  __shared__ uint32_t red[8];
  __shared__ uint32_t amax_sh, ok_sh;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint32_t m = 0;
  {
    int t = 0;
    for (; t + 1 < R; t += 2)
      m = max(m, amax_pass2(reinterpret_cast<const float4 *>(a.x[t]), reinterpret_cast<const float4 *>(a.x[t + 1]), n4,
                            tid, stride));
    if (t < R) m = max(m, amax_pass(reinterpret_cast<const float4 *>(a.x[t]), n4, tid, stride));
  }
  m = block_max_u32<256>(m, red);
  if (threadIdx.x == 0) {
    if (m) atomicMax(ws, m);
    if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws + 1) : "memory");
    uint32_t ok = 1;
    const long long t0 = clock64();
    while (ld_acquire_gpu(ws + 1) < gridDim.x) {
      if (clock64() - t0 > wait_budget) {
        ok = 0;
        set_status(status, GIFT_ERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    amax_sh = ld_acquire_gpu(ws);
    ok_sh = ok;
  }
  __syncthreads();
  if (!ok_sh) return;
  const float amax = __uint_as_float(amax_sh);
  const ScalePair sp = scale_pair(amax, fmax_of<F>());
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
    for (int t = 0; t < R; ++t) {
      a.scale[t][0] = sp.s;
      if (a.amax_out[t]) a.amax_out[t][0] = amax;
    }
    if (shared_out) shared_out[0] = amax;
  }
  int t = R - 1;
  for (; t >= 1; t -= 2)
    pack_pass2<F>(reinterpret_cast<const float4 *>(a.x[t]), reinterpret_cast<uint32_t *>(a.codes[t]),
                  reinterpret_cast<const float4 *>(a.x[t - 1]), reinterpret_cast<uint32_t *>(a.codes[t - 1]), n4, tid,
                  stride, sp);
  if (t == 0)
    pack_pass<F>(reinterpret_cast<const float4 *>(a.x[0]), reinterpret_cast<uint32_t *>(a.codes[0]), n4, tid, stride,
                 sp);
}

// =====================================================================================
// FP32 "format": codes are the values themselves (lossless path); residual becomes 0.
// =====================================================================================
template <bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_pack_f32(const float *__restrict__ x, float *__restrict__ r, size_t n,
                                                  float *__restrict__ out, float *__restrict__ tout) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = x[i];
    if (RES) {
      v = __fadd_rn(v, r[i]);
      r[i] = 0.0f;
    }
    out[i] = v;
    if (TOUT) tout[i] = v;
  }
}

// =====================================================================================
// 128 x 128 block scaling, one CTA per tile (amax, scale and pack in one pass).
// Thread layout: warp w holds rows w + 8k (k < 16), lane l columns 4l..4l+3.
// MODE 0: pack; MODE 1: amax only (atomicMax into amax_out[tile]); MODE 2: count hits.
// =====================================================================================
template <int F, int MODE, bool VEC, bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_block128(const float *__restrict__ x, float *__restrict__ r, int d_out,
                                                  int d_in, const float *__restrict__ amax_in,
                                                  uint8_t *__restrict__ codes, float *__restrict__ scales,
                                                  float *__restrict__ amax_out, float *__restrict__ tout,
                                                  unsigned long long *__restrict__ counts, int *status) {
  __shared__ uint32_t red[8];
  const int nbc = (d_in + kBlock - 1) / kBlock;
  const int tile = blockIdx.y * nbc + blockIdx.x;
  const int r0 = blockIdx.y * kBlock, c0 = blockIdx.x * kBlock;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int col = c0 + 4 * l;
  float v[16][4];
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = r0 + w + 8 * k;
    const size_t base = (size_t)row * d_in + col;
    if (VEC) {
      if (row < d_out && col < d_in) {
        float4 a = *reinterpret_cast<const float4 *>(x + base);
        if (RES) a = add4(a, *reinterpret_cast<const float4 *>(r + base));
        v[k][0] = a.x; v[k][1] = a.y; v[k][2] = a.z; v[k][3] = a.w;
      } else {
        v[k][0] = v[k][1] = v[k][2] = v[k][3] = 0.0f;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a = 0.0f;
        if (row < d_out && col + e < d_in) {
          a = x[base + e];
          if (RES) a = __fadd_rn(a, r[base + e]);
        }
        v[k][e] = a;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) m = max(m, abs_bits(v[k][e]));
  }
  m = block_max_u32<256>(m, red);
  if (MODE == 1) {
    if (threadIdx.x == 0) {
      atomicMax(reinterpret_cast<uint32_t *>(amax_out) + tile, m);
      if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
    }
    return;
  }
  float amax = __uint_as_float(m);
  if (MODE == 0 && amax_in) amax = amax_in[tile];
  const ScalePair sp = scale_pair(amax, fmax_of<F>());
  if (threadIdx.x == 0) {
    if (m >= 0x7F800000u || !(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
    if (MODE == 0) {
      scales[tile] = sp.s;
      if (amax_out) amax_out[tile] = amax;
    }
  }
  uint32_t up = 0, lo = 0, cnt = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int row = r0 + w + 8 * k;
    if (row >= d_out || col >= d_in) continue;
    const size_t base = (size_t)row * d_in + col;
    const uint32_t c = pack4_fp8<F>(__fmul_rn(v[k][0], sp.m), __fmul_rn(v[k][1], sp.m),
                                    __fmul_rn(v[k][2], sp.m), __fmul_rn(v[k][3], sp.m));
    if (MODE == 2) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (col + e < d_in) {
          const uint32_t mag = (c >> (8 * e)) & 0x7Fu;
          up += (mag == maxcode_of<F>());
          lo += (mag == 0u && v[k][e] != 0.0f);
          ++cnt;
        }
      }
      continue;
    }
    if (VEC) {
      *reinterpret_cast<uint32_t *>(codes + base) = c;
      if (TOUT) *reinterpret_cast<float4 *>(tout + base) = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
      if (RES) {
        float4 e;
        e.x = __fsub_rn(v[k][0], __fmul_rn(dec_fp8<F>(c & 0xFF), sp.s));
        e.y = __fsub_rn(v[k][1], __fmul_rn(dec_fp8<F>((c >> 8) & 0xFF), sp.s));
        e.z = __fsub_rn(v[k][2], __fmul_rn(dec_fp8<F>((c >> 16) & 0xFF), sp.s));
        e.w = __fsub_rn(v[k][3], __fmul_rn(dec_fp8<F>(c >> 24), sp.s));
        *reinterpret_cast<float4 *>(r + base) = e;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (col + e >= d_in) continue;
        const uint32_t ce = (c >> (8 * e)) & 0xFFu;
        codes[base + e] = (uint8_t)ce;
        if (TOUT) tout[base + e] = v[k][e];
        if (RES) r[base + e] = __fsub_rn(v[k][e], __fmul_rn(dec_fp8<F>(ce), sp.s));
      }
    }
  }
  if (MODE == 2) {
    up = warp_add_u32(up);
    lo = warp_add_u32(lo);
    cnt = warp_add_u32(cnt);
    if (l == 0 && cnt) {
      atomicAdd(counts + 0, (unsigned long long)up);
      atomicAdd(counts + 1, (unsigned long long)lo);
      atomicAdd(counts + 2, (unsigned long long)cnt);
    }
  }
}

// =====================================================================================
// NVFP4 pack.  Vector path: a quad of threads holds one group of 16 consecutive elements
// (one float4 each) and shares the group amax by shuffles.  Needs n % 16 == 0.
// =====================================================================================
template <bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_pack_nvfp4_vec(const float *__restrict__ x, float *__restrict__ r,
                                                        size_t n, const float *__restrict__ amax_ptr,
                                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ bscale,
                                                        float *__restrict__ tscale_out, float *__restrict__ amax_out,
                                                        float *__restrict__ tout, int *status) {
  const float amax = *amax_ptr;
  const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
    tscale_out[0] = s_t;
    if (amax_out) amax_out[0] = amax;
  }
  const size_t n4 = n >> 2;
  const float4 *x4 = reinterpret_cast<const float4 *>(x);
  float4 *r4 = reinterpret_cast<float4 *>(r);
  float4 *t4 = reinterpret_cast<float4 *>(tout);
  uint16_t *c2 = reinterpret_cast<uint16_t *>(codes);
  const size_t warp0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) & ~(size_t)31;
  const int lane = threadIdx.x & 31;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t base = warp0; base < n4; base += stride) {
    const size_t i = base + lane;
    const bool ok = i < n4;   // n4 % 4 == 0, so a quad is all in or all out
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
      v = x4[i];
      if (RES) v = add4(v, r4[i]);
    }
    uint32_t gm = max(max(abs_bits(v.x), abs_bits(v.y)), max(abs_bits(v.z), abs_bits(v.w)));
    gm = max(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 1));
    gm = max(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 2));
    if (!ok) continue;
    const Nv4Group g = nvfp4_group(__uint_as_float(gm), s_t);
    if (TOUT) t4[i] = v;
    const uint32_t c = pack4_e2m1(__fmul_rn(v.x, g.r), __fmul_rn(v.y, g.r), __fmul_rn(v.z, g.r),
                                  __fmul_rn(v.w, g.r));
    c2[i] = (uint16_t)c;
    if ((lane & 3) == 0) bscale[i >> 2] = g.e_code;
    if (RES) {
      const float ev = dec_e4m3(g.e_code);
      float4 e;
      e.x = __fsub_rn(v.x, nvfp4_deq(c & 0xF, ev, s_t));
      e.y = __fsub_rn(v.y, nvfp4_deq((c >> 4) & 0xF, ev, s_t));
      e.z = __fsub_rn(v.z, nvfp4_deq((c >> 8) & 0xF, ev, s_t));
      e.w = __fsub_rn(v.w, nvfp4_deq((c >> 12) & 0xF, ev, s_t));
      r4[i] = e;
    }
  }
}

// Scalar NVFP4 path: one thread per group of 16.
template <bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_pack_nvfp4_scalar(const float *__restrict__ x, float *__restrict__ r,
                                                           size_t n, const float *__restrict__ amax_ptr,
                                                           uint8_t *__restrict__ codes, uint8_t *__restrict__ bscale,
                                                           float *__restrict__ tscale_out,
                                                           float *__restrict__ amax_out, float *__restrict__ tout,
                                                           int *status) {
  const float amax = *amax_ptr;
  const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
    tscale_out[0] = s_t;
    if (amax_out) amax_out[0] = amax;
  }
  const size_t ng = n / kNvGroup;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t gi = (size_t)blockIdx.x * blockDim.x + threadIdx.x; gi < ng; gi += stride) {
    float v[16];
    uint32_t gm = 0;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      v[e] = x[gi * 16 + e];
      if (RES) v[e] = __fadd_rn(v[e], r[gi * 16 + e]);
      gm = max(gm, abs_bits(v[e]));
    }
    const Nv4Group g = nvfp4_group(__uint_as_float(gm), s_t);
    const float ev = dec_e4m3(g.e_code);
    bscale[gi] = g.e_code;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(v[8 * h + e], g.r);
      const uint32_t c = pack8_e2m1(y);
#pragma unroll
      for (int b = 0; b < 4; ++b) codes[gi * 8 + 4 * h + b] = (uint8_t)(c >> (8 * b));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const size_t idx = gi * 16 + 8 * h + e;
        if (TOUT) tout[idx] = v[8 * h + e];
        if (RES) r[idx] = __fsub_rn(v[8 * h + e], nvfp4_deq((c >> (4 * e)) & 0xF, ev, s_t));
      }
    }
  }
}

// =====================================================================================
// boundary-hit counting with the tensor scale (amax read from *amax_ptr).
// =====================================================================================
template <int F, bool VEC>
__global__ void __launch_bounds__(256) k_hits_tensor(const float *__restrict__ x, size_t n,
                                                     const float *__restrict__ amax_ptr,
                                                     unsigned long long *__restrict__ counts) {
  const float amax = *amax_ptr;
  const ScalePair sp = scale_pair(amax, fmax_of<F>());
  uint32_t up = 0, lo = 0, cnt = 0;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t done = 0;
  if (VEC) {
    const size_t n4 = n >> 2;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    for (size_t i = tid; i < n4; i += stride) {
      const float4 v = x4[i];
      const uint32_t c = pack4_fp8<F>(__fmul_rn(v.x, sp.m), __fmul_rn(v.y, sp.m), __fmul_rn(v.z, sp.m),
                                      __fmul_rn(v.w, sp.m));
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t mag = (c >> (8 * e)) & 0x7Fu;
        up += (mag == maxcode_of<F>());
        lo += (mag == 0u && vv[e] != 0.0f);
      }
      cnt += 4;
    }
    done = n4 << 2;
  }
  for (size_t i = done + tid; i < n; i += stride) {
    const float v = x[i];
    const uint32_t mag = pack1_fp8<F>(__fmul_rn(v, sp.m)) & 0x7Fu;
    up += (mag == maxcode_of<F>());
    lo += (mag == 0u && v != 0.0f);
    ++cnt;
  }
  up = warp_add_u32(up);
  lo = warp_add_u32(lo);
  cnt = warp_add_u32(cnt);
  if ((threadIdx.x & 31) == 0 && cnt) {
    atomicAdd(counts + 0, (unsigned long long)up);
    atomicAdd(counts + 1, (unsigned long long)lo);
    atomicAdd(counts + 2, (unsigned long long)cnt);
  }
}

// =====================================================================================
// 1-D block scaling: one FP32 scale per kBlock1d = 512 consecutive elements of the row-major
// tensor, the last block shorter (the per-block Euclidean baseline of the experiments, block
// size 512).  One warp per block: VEC, lane l holds elements 4(l + 32u) .. +3 (u < 4) as
// float4, every load and store coalesced; otherwise lane l holds elements l + 32j (j < 16).
// MODE 0: pack (amax_in per block overrides the block's own); MODE 1: amax only
// (atomicMax into amax_out[block]); MODE 2: count boundary hits.  Per element the
// arithmetic is that of the per-tensor pack.
// =====================================================================================
template <int F, int MODE, bool VEC, bool RES, bool TOUT>
__global__ void __launch_bounds__(256) k_block512(const float *__restrict__ x, float *__restrict__ r, size_t n,
                                                  const float *__restrict__ amax_in, uint8_t *__restrict__ codes,
                                                  float *__restrict__ scales, float *__restrict__ amax_out,
                                                  float *__restrict__ tout, unsigned long long *__restrict__ counts,
                                                  int *status) {
  const int lane = threadIdx.x & 31;
  const size_t nb = (n + kBlock1d - 1) / kBlock1d;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  uint32_t up = 0, lo = 0, cnt = 0;
  for (size_t b = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nb; b += warps) {
    const size_t e0 = b * kBlock1d;
    const size_t len = min((size_t)kBlock1d, n - e0);
    float v[16];
    uint32_t m = 0;
    if (VEC) {   // n % 4 == 0, 16-byte aligned x (and r)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const size_t i = 4 * (lane + 32 * u);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < len) {
          a = *reinterpret_cast<const float4 *>(x + e0 + i);
          if (RES) a = add4(a, *reinterpret_cast<const float4 *>(r + e0 + i));
        }
        v[4 * u] = a.x; v[4 * u + 1] = a.y; v[4 * u + 2] = a.z; v[4 * u + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const size_t i = lane + 32 * j;
        float a = 0.0f;
        if (i < len) {
          a = x[e0 + i];
          if (RES) a = __fadd_rn(a, r[e0 + i]);
        }
        v[j] = a;
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) m = max(m, abs_bits(v[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (MODE == 1) {
      if (lane == 0) {
        atomicMax(reinterpret_cast<uint32_t *>(amax_out) + b, m);
        if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
      }
      continue;
    }
    float amax = __uint_as_float(m);
    if (MODE == 0 && amax_in) amax = amax_in[b];
    const ScalePair sp = scale_pair(amax, fmax_of<F>());
    if (lane == 0) {
      if (m >= 0x7F800000u || !(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
      if (MODE == 0) {
        scales[b] = sp.s;
        if (amax_out) amax_out[b] = amax;
      }
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t c = pack4_fp8<F>(__fmul_rn(v[4 * g], sp.m), __fmul_rn(v[4 * g + 1], sp.m),
                                      __fmul_rn(v[4 * g + 2], sp.m), __fmul_rn(v[4 * g + 3], sp.m));
      if (VEC) {
        const size_t i = 4 * (lane + 32 * g);
        if (i >= len) continue;
        if (MODE == 2) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t mag = (c >> (8 * e)) & 0x7Fu;
            up += (mag == maxcode_of<F>());
            lo += (mag == 0u && v[4 * g + e] != 0.0f);
            ++cnt;
          }
          continue;
        }
        *reinterpret_cast<uint32_t *>(codes + e0 + i) = c;
        if (TOUT) *reinterpret_cast<float4 *>(tout + e0 + i) = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        if (RES) {
          float4 e;
          e.x = __fsub_rn(v[4 * g], __fmul_rn(dec_fp8<F>(c & 0xFF), sp.s));
          e.y = __fsub_rn(v[4 * g + 1], __fmul_rn(dec_fp8<F>((c >> 8) & 0xFF), sp.s));
          e.z = __fsub_rn(v[4 * g + 2], __fmul_rn(dec_fp8<F>((c >> 16) & 0xFF), sp.s));
          e.w = __fsub_rn(v[4 * g + 3], __fmul_rn(dec_fp8<F>(c >> 24), sp.s));
          *reinterpret_cast<float4 *>(r + e0 + i) = e;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * g + e;
          const size_t i = lane + 32 * j;
          if (i >= len) continue;
          const uint32_t ce = (c >> (8 * e)) & 0xFFu;
          if (MODE == 2) {
            up += ((ce & 0x7Fu) == maxcode_of<F>());
            lo += ((ce & 0x7Fu) == 0u && v[j] != 0.0f);
            ++cnt;
            continue;
          }
          codes[e0 + i] = (uint8_t)ce;
          if (TOUT) tout[e0 + i] = v[j];
          if (RES) r[e0 + i] = __fsub_rn(v[j], __fmul_rn(dec_fp8<F>(ce), sp.s));
        }
      }
    }
  }
  if (MODE == 2) {
    up = warp_add_u32(up);
    lo = warp_add_u32(lo);
    cnt = warp_add_u32(cnt);
    if (lane == 0 && cnt) {
      atomicAdd(counts + 0, (unsigned long long)up);
      atomicAdd(counts + 1, (unsigned long long)lo);
      atomicAdd(counts + 2, (unsigned long long)cnt);
    }
  }
}

// =====================================================================================
// Replica reduce: out = (deq_0 + deq_1 + ... + deq_{R-1}) / R, left to right in FP32.
// Vector path: 16 elements per thread (one 16-byte code load per replica).
// =====================================================================================
// SC: 0 per tensor, 1 per 128 x 128 tile, 2 per 512 consecutive elements
template <int SC>
__device__ __forceinline__ float replica_scale(const ReduceArgs &a, int rr, size_t e0, int d_in, int nbc) {
  const float *s = reinterpret_cast<const float *>(a.scales[rr]);
  if (SC == 0) return s[0];
  if (SC == 2) return s[e0 / kBlock1d];
  const size_t row = e0 / (size_t)d_in;
  const int col = (int)(e0 - row * (size_t)d_in);
  return s[(row / kBlock) * nbc + col / kBlock];
}

template <int F, int SC>
__global__ void __launch_bounds__(256) k_reduce_fp8_vec(ReduceArgs a, int R, size_t n, int d_in,
                                                        float *__restrict__ out) {
  const size_t n16 = n >> 4;
  const int nbc = (d_in + kBlock - 1) / kBlock;
  const float div = (float)R;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    float acc[16];
    const size_t e0 = i << 4;
    // the replicas' code chunks are loaded 8 at a time (8 loads in flight per thread), then
    // added in replica order
    for (int r0 = 0; r0 < R; r0 += 8) {
      uint4 cc[8];
      float sc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (r0 + u < R) {
          cc[u] = __ldcs(reinterpret_cast<const uint4 *>(a.codes[r0 + u]) + i);
          sc[u] = replica_scale<SC>(a, r0 + u, e0, d_in, nbc);
        }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (r0 + u < R) {
          const uint32_t w[4] = {cc[u].x, cc[u].y, cc[u].z, cc[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float d = __fmul_rn(dec_fp8<F>((w[q] >> (8 * b)) & 0xFFu), sc[u]);
              acc[4 * q + b] = (r0 + u == 0) ? d : __fadd_rn(acc[4 * q + b], d);
            }
          }
        }
    }
    float4 *o = reinterpret_cast<float4 *>(out + e0);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = make_float4(__fdiv_rn(acc[4 * q], div), __fdiv_rn(acc[4 * q + 1], div),
                         __fdiv_rn(acc[4 * q + 2], div), __fdiv_rn(acc[4 * q + 3], div));
  }
}

// NVFP4 vector path: one group of 16 per thread (8 code bytes + 1 scale byte per replica).
__global__ void __launch_bounds__(256) k_reduce_nvfp4_vec(ReduceArgs a, int R, size_t n,
                                                          float *__restrict__ out) {
  const size_t ng = n >> 4;
  const float div = (float)R;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < ng; g += stride) {
    float acc[16];
    for (int rr = 0; rr < R; ++rr) {
      const uint2 c = reinterpret_cast<const uint2 *>(a.codes[rr])[g];
      const float ev = dec_e4m3(reinterpret_cast<const uint8_t *>(a.scales[rr])[g]);
      const float st = a.tscales[rr][0];
      const uint32_t w[2] = {c.x, c.y};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const float d = nvfp4_deq((w[q] >> (4 * b)) & 0xFu, ev, st);
          acc[8 * q + b] = (rr == 0) ? d : __fadd_rn(acc[8 * q + b], d);
        }
      }
    }
    float4 *o = reinterpret_cast<float4 *>(out + (g << 4));
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = make_float4(__fdiv_rn(acc[4 * q], div), __fdiv_rn(acc[4 * q + 1], div),
                         __fdiv_rn(acc[4 * q + 2], div), __fdiv_rn(acc[4 * q + 3], div));
  }
}

// Generic scalar path (any alignment, any format); element range [start, n).
// FMTK: 0 E4M3, 1 E5M2, 2 NVFP4, 3 F32.
template <int FMTK, int SC>
__global__ void __launch_bounds__(256) k_reduce_scalar(ReduceArgs a, int R, size_t start, size_t n, int d_in,
                                                       float *__restrict__ out) {
  const int nbc = (d_in + kBlock - 1) / kBlock;
  const float div = (float)R;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t e = start + (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    float acc = 0.0f;
    for (int rr = 0; rr < R; ++rr) {
      float d;
      if (FMTK == 3) {
        d = reinterpret_cast<const float *>(a.codes[rr])[e];
      } else if (FMTK == 2) {
        const uint8_t byte = reinterpret_cast<const uint8_t *>(a.codes[rr])[e >> 1];
        const uint32_t c = (e & 1) ? (byte >> 4) : (byte & 0xF);
        const float ev = dec_e4m3(reinterpret_cast<const uint8_t *>(a.scales[rr])[e >> 4]);
        d = nvfp4_deq(c, ev, a.tscales[rr][0]);
      } else {
        const uint8_t c = reinterpret_cast<const uint8_t *>(a.codes[rr])[e];
        const float s = replica_scale<SC>(a, rr, e, d_in, nbc);
        d = __fmul_rn(FMTK == 0 ? dec_e4m3(c) : dec_e5m2(c), s);
      }
      acc = (rr == 0) ? d : __fadd_rn(acc, d);
    }
    out[e] = __fdiv_rn(acc, div);
  }
}

// F32 vector path: 4 elements per thread.
__global__ void __launch_bounds__(256) k_reduce_f32_vec(ReduceArgs a, int R, size_t n, float *__restrict__ out) {
  const size_t n4 = n >> 2;
  const float div = (float)R;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 acc = reinterpret_cast<const float4 *>(a.codes[0])[i];
    for (int rr = 1; rr < R; ++rr) acc = add4(acc, reinterpret_cast<const float4 *>(a.codes[rr])[i]);
    reinterpret_cast<float4 *>(out)[i] =
        make_float4(__fdiv_rn(acc.x, div), __fdiv_rn(acc.y, div), __fdiv_rn(acc.z, div), __fdiv_rn(acc.w, div));
  }
}

// =====================================================================================
// launchers
// =====================================================================================
static int stream_grid(const Launch &L, size_t work, int per_cta) {
  size_t g = (work + per_cta - 1) / per_cta;
  const size_t cap = (size_t)L.sms * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

cudaError_t launch_amax(const Launch &L, const float *x, const float *r, size_t n, float *amax_accum) {
  if (!r && aligned16(x) && n % 4 == 0) {   // the streaming multi-tensor kernel, one tensor
    MultiArgs m;
    m.x[0] = x;
    m.amax_bits[0] = reinterpret_cast<uint32_t *>(amax_accum);
    return launch_amax_multi(L, m, 1, n);
  }
  const bool vec = aligned16(x) && (r == nullptr || aligned16(r));
  const int grid = stream_grid(L, (n + 3) / 4, 256);
  uint32_t *ab = reinterpret_cast<uint32_t *>(amax_accum);
  if (vec) {
    if (r) k_amax<true, true><<<grid, 256, 0, L.stream>>>(x, r, n, ab, L.status);
    else k_amax<true, false><<<grid, 256, 0, L.stream>>>(x, r, n, ab, L.status);
  } else {
    if (r) k_amax<false, true><<<grid, 256, 0, L.stream>>>(x, r, n, ab, L.status);
    else k_amax<false, false><<<grid, 256, 0, L.stream>>>(x, r, n, ab, L.status);
  }
  return cudaGetLastError();
}

template <int F, bool VEC>
static void pack_tensor_dispatch(const Launch &L, int grid, const float *x, float *r, size_t n, const float *amax,
                                 uint8_t *codes, float *scale, float *amax_out, float *tout) {
#define PT(RS, TO) k_pack_tensor<F, VEC, RS, TO><<<grid, 256, 0, L.stream>>>(x, r, n, amax, codes, scale, amax_out, tout, L.status)
  if (r) { if (tout) PT(true, true); else PT(true, false); }
  else { if (tout) PT(false, true); else PT(false, false); }
#undef PT
}

cudaError_t launch_pack_tensor(const Launch &L, int fmt, const float *x, float *r, size_t n, const float *amax,
                               uint8_t *codes, float *scale, float *amax_out, float *tout) {
  if (!r && !tout && aligned16(x) && n % 4 == 0 && ((uintptr_t)codes & 3u) == 0) {   // one tensor, streaming
    MultiArgs m;
    m.x[0] = x;
    m.codes[0] = codes;
    m.scale[0] = scale;
    m.amax_in[0] = amax;
    m.amax_out[0] = amax_out;
    return launch_pack_tensor_multi(L, fmt, m, 1, n);
  }
  const bool vec = aligned16(x) && (!r || aligned16(r)) && (!tout || aligned16(tout)) &&
                   (((uintptr_t)codes & 3u) == 0);
  const int grid = stream_grid(L, (n + 3) / 4, 256);
  if (fmt == GIFT_FMT_E4M3) {
    if (vec) pack_tensor_dispatch<FMT_E4M3, true>(L, grid, x, r, n, amax, codes, scale, amax_out, tout);
    else pack_tensor_dispatch<FMT_E4M3, false>(L, grid, x, r, n, amax, codes, scale, amax_out, tout);
  } else {
    if (vec) pack_tensor_dispatch<FMT_E5M2, true>(L, grid, x, r, n, amax, codes, scale, amax_out, tout);
    else pack_tensor_dispatch<FMT_E5M2, false>(L, grid, x, r, n, amax, codes, scale, amax_out, tout);
  }
  return cudaGetLastError();
}

bool multi_ok(const MultiArgs &a, int R, size_t n, bool pack) {
  if (R < 1 || R > kMaxReplicas || n % 4) return false;
  for (int t = 0; t < R; ++t) {
    if (!aligned16(a.x[t])) return false;
    if (pack && ((uintptr_t)a.codes[t] & 3u)) return false;
  }
  return true;
}

cudaError_t launch_amax_multi(const Launch &L, const MultiArgs &a, int R, size_t n) {
  const int grid = stream_grid(L, n / 4, 1024);
  k_amax_multi<<<grid, 256, 0, L.stream>>>(a, R, n / 4, L.status);
  return cudaGetLastError();
}

cudaError_t launch_pack_tensor_multi(const Launch &L, int fmt, const MultiArgs &a, int R, size_t n) {
  const int grid = stream_grid(L, n / 4, 1024);
  if (fmt == GIFT_FMT_E4M3) k_pack_tensor_multi<FMT_E4M3><<<grid, 256, 0, L.stream>>>(a, R, n / 4, L.status);
  else k_pack_tensor_multi<FMT_E5M2><<<grid, 256, 0, L.stream>>>(a, R, n / 4, L.status);
  return cudaGetLastError();
}

cudaError_t launch_encode_shared(const Launch &L, int fmt, const MultiArgs &a, int R, size_t n, uint32_t *ws,
                                 float *shared_out) {
  const void *kern = (fmt == GIFT_FMT_E4M3) ? reinterpret_cast<const void *>(&k_encode_shared<FMT_E4M3>)
                                            : reinterpret_cast<const void *>(&k_encode_shared<FMT_E5M2>);
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = stream_grid(L, n / 4, 1024);
  if (grid > per_sm * L.sms) grid = per_sm * L.sms;   // every CTA resident: the barrier needs it
  MultiArgs args_a = a;
  int args_r = R;
  size_t n4 = n / 4;
  int *st = L.status;
  long long budget = L.barrier_wait;
  void *args[] = {&args_a, &args_r, &n4, &ws, &shared_out, &budget, &st};
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kern, args);
}

cudaError_t launch_pack_f32(const Launch &L, const float *x, float *r, size_t n, float *out, float *tout) {
  const int grid = stream_grid(L, n, 256);
  if (r) {
    if (tout) k_pack_f32<true, true><<<grid, 256, 0, L.stream>>>(x, r, n, out, tout);
    else k_pack_f32<true, false><<<grid, 256, 0, L.stream>>>(x, r, n, out, tout);
  } else {
    if (tout) k_pack_f32<false, true><<<grid, 256, 0, L.stream>>>(x, r, n, out, tout);
    else k_pack_f32<false, false><<<grid, 256, 0, L.stream>>>(x, r, n, out, tout);
  }
  return cudaGetLastError();
}

template <int F, int MODE, bool VEC>
static void block_dispatch(const Launch &L, dim3 grid, const float *x, float *r, int d_out, int d_in,
                           const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                           unsigned long long *counts) {
#define BK(RS, TO) k_block128<F, MODE, VEC, RS, TO><<<grid, 256, 0, L.stream>>>(x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts, L.status)
  if (r) { if (tout) BK(true, true); else BK(true, false); }
  else { if (tout) BK(false, true); else BK(false, false); }
#undef BK
}

template <int F, int MODE>
static void block_dispatch_v(const Launch &L, bool vec, dim3 grid, const float *x, float *r, int d_out, int d_in,
                             const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                             unsigned long long *counts) {
  if (vec) block_dispatch<F, MODE, true>(L, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
  else block_dispatch<F, MODE, false>(L, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
}

template <int F>
static void block_modes(const Launch &L, int mode, bool vec, dim3 grid, const float *x, float *r, int d_out,
                        int d_in, const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                        unsigned long long *counts) {
  if (mode == 0) block_dispatch_v<F, 0>(L, vec, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
  else if (mode == 1) block_dispatch_v<F, 1>(L, vec, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
  else block_dispatch_v<F, 2>(L, vec, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
}

cudaError_t launch_block128(const Launch &L, int fmt, int mode, const float *x, float *r, int d_out, int d_in,
                            const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                            unsigned long long *counts) {
  const bool vec = (d_in % 4 == 0) && aligned16(x) && (!r || aligned16(r)) && (!tout || aligned16(tout)) &&
                   (((uintptr_t)codes & 3u) == 0);
  dim3 grid((d_in + kBlock - 1) / kBlock, (d_out + kBlock - 1) / kBlock);
  if (fmt == GIFT_FMT_E4M3) block_modes<FMT_E4M3>(L, mode, vec, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
  else block_modes<FMT_E5M2>(L, mode, vec, grid, x, r, d_out, d_in, amax_in, codes, scales, amax_out, tout, counts);
  return cudaGetLastError();
}

cudaError_t launch_pack_nvfp4(const Launch &L, const float *x, float *r, size_t n, const float *amax,
                              uint8_t *codes, uint8_t *bscale, float *tscale, float *amax_out, float *tout) {
  const bool vec = aligned16(x) && (!r || aligned16(r)) && (!tout || aligned16(tout)) &&
                   (((uintptr_t)codes & 1u) == 0);
  if (vec) {
    const int grid = stream_grid(L, n / 4, 256);
#define NV_V(RS, TO) k_pack_nvfp4_vec<RS, TO><<<grid, 256, 0, L.stream>>>(x, r, n, amax, codes, bscale, tscale, amax_out, tout, L.status)
    if (r) { if (tout) NV_V(true, true); else NV_V(true, false); }
    else { if (tout) NV_V(false, true); else NV_V(false, false); }
#undef NV_V
  } else {
    const int grid = stream_grid(L, n / 16, 256);
#define NV_S(RS, TO) k_pack_nvfp4_scalar<RS, TO><<<grid, 256, 0, L.stream>>>(x, r, n, amax, codes, bscale, tscale, amax_out, tout, L.status)
    if (r) { if (tout) NV_S(true, true); else NV_S(true, false); }
    else { if (tout) NV_S(false, true); else NV_S(false, false); }
#undef NV_S
  }
  return cudaGetLastError();
}

cudaError_t launch_hits_tensor(const Launch &L, int fmt, const float *x, size_t n, const float *amax,
                               unsigned long long *counts) {
  const bool vec = aligned16(x);
  const int grid = stream_grid(L, (n + 3) / 4, 256);
  if (fmt == GIFT_FMT_E4M3) {
    if (vec) k_hits_tensor<FMT_E4M3, true><<<grid, 256, 0, L.stream>>>(x, n, amax, counts);
    else k_hits_tensor<FMT_E4M3, false><<<grid, 256, 0, L.stream>>>(x, n, amax, counts);
  } else {
    if (vec) k_hits_tensor<FMT_E5M2, true><<<grid, 256, 0, L.stream>>>(x, n, amax, counts);
    else k_hits_tensor<FMT_E5M2, false><<<grid, 256, 0, L.stream>>>(x, n, amax, counts);
  }
  return cudaGetLastError();
}

template <int F, int SC>
static void reduce_fp8(const Launch &L, const ReduceArgs &a, int R, size_t n, size_t done, int d_in, float *out,
                       bool vec) {
  if (vec) k_reduce_fp8_vec<F, SC><<<stream_grid(L, n / 16, 256), 256, 0, L.stream>>>(a, R, n, d_in, out);
  if (done < n)
    k_reduce_scalar<F == FMT_E4M3 ? 0 : 1, SC><<<stream_grid(L, n - done, 256), 256, 0, L.stream>>>(a, R, done, n,
                                                                                                      d_in, out);
}

cudaError_t launch_reduce(const Launch &L, const ReduceArgs &a, int R, int fmt, int scaling, int d_out, int d_in,
                          float *out) {
  const size_t n = (size_t)d_out * d_in;
  bool vec = aligned16(out);
  for (int rr = 0; rr < R && vec; ++rr) vec = aligned16(a.codes[rr]);
  size_t done = 0;
  if (fmt == GIFT_FMT_F32) {
    if (vec) {
      k_reduce_f32_vec<<<stream_grid(L, n / 4, 256), 256, 0, L.stream>>>(a, R, n, out);
      done = (n / 4) * 4;
    }
    if (done < n) k_reduce_scalar<3, 0><<<stream_grid(L, n - done, 256), 256, 0, L.stream>>>(a, R, done, n, d_in, out);
  } else if (fmt == GIFT_FMT_NVFP4) {
    bool v8 = aligned16(out);
    for (int rr = 0; rr < R && v8; ++rr) v8 = (((uintptr_t)a.codes[rr]) & 7u) == 0;
    if (v8) {
      k_reduce_nvfp4_vec<<<stream_grid(L, n / 16, 256), 256, 0, L.stream>>>(a, R, n, out);
      done = n;   // NVFP4 needs d_in % 16 == 0, so n % 16 == 0
    }
    if (done < n) k_reduce_scalar<2, 0><<<stream_grid(L, n - done, 256), 256, 0, L.stream>>>(a, R, done, n, d_in, out);
  } else {
    // the vector path looks a scale up once per 16 elements: a group of 16 must not cross a
    // 128-column tile edge (block 512 groups never cross a block)
    const int sc = (scaling == GIFT_SCALE_BLOCK128) ? 1 : (scaling == GIFT_SCALE_BLOCK512) ? 2 : 0;
    vec = vec && (sc != 1 || d_in % 16 == 0);
    if (vec) done = (n / 16) * 16;
    if (fmt == GIFT_FMT_E4M3) {
      if (sc == 0) reduce_fp8<FMT_E4M3, 0>(L, a, R, n, done, d_in, out, vec);
      else if (sc == 1) reduce_fp8<FMT_E4M3, 1>(L, a, R, n, done, d_in, out, vec);
      else reduce_fp8<FMT_E4M3, 2>(L, a, R, n, done, d_in, out, vec);
    } else {
      if (sc == 0) reduce_fp8<FMT_E5M2, 0>(L, a, R, n, done, d_in, out, vec);
      else if (sc == 1) reduce_fp8<FMT_E5M2, 1>(L, a, R, n, done, d_in, out, vec);
      else reduce_fp8<FMT_E5M2, 2>(L, a, R, n, done, d_in, out, vec);
    }
  }
  return cudaGetLastError();
}

template <int F, int MODE>
static void block512_launch(const Launch &L, bool vec, const float *x, float *r, size_t n, const float *amax_in,
                            uint8_t *codes, float *scales, float *amax_out, float *tout,
                            unsigned long long *counts) {
  const size_t nb = (n + kBlock1d - 1) / kBlock1d;
  const int grid = stream_grid(L, nb, 8);   // 8 warps, one block each per step
#define GIFT_B512(V, RS, TO) \
  k_block512<F, MODE, V, RS, TO><<<grid, 256, 0, L.stream>>>(x, r, n, amax_in, codes, scales, amax_out, tout, counts, L.status)
  if (vec) {
    if (r) { if (tout) GIFT_B512(true, true, true); else GIFT_B512(true, true, false); }
    else { if (tout) GIFT_B512(true, false, true); else GIFT_B512(true, false, false); }
  } else {
    if (r) { if (tout) GIFT_B512(false, true, true); else GIFT_B512(false, true, false); }
    else { if (tout) GIFT_B512(false, false, true); else GIFT_B512(false, false, false); }
  }
#undef GIFT_B512
}

cudaError_t launch_block512(const Launch &L, int fmt, int mode, const float *x, float *r, size_t n,
                            const float *amax_in, uint8_t *codes, float *scales, float *amax_out, float *tout,
                            unsigned long long *counts) {
  const bool vec = n % 4 == 0 && aligned16(x) && (!r || aligned16(r)) && (!tout || aligned16(tout)) &&
                   (mode != 0 || (((uintptr_t)codes) & 3u) == 0);
  if (fmt == GIFT_FMT_E4M3) {
    if (mode == 0) block512_launch<FMT_E4M3, 0>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
    else if (mode == 1) block512_launch<FMT_E4M3, 1>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
    else block512_launch<FMT_E4M3, 2>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
  } else {
    if (mode == 0) block512_launch<FMT_E5M2, 0>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
    else if (mode == 1) block512_launch<FMT_E5M2, 1>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
    else block512_launch<FMT_E5M2, 2>(L, vec, x, r, n, amax_in, codes, scales, amax_out, tout, counts);
  }
  return cudaGetLastError();
}

cudaError_t launch_hits_multi(const Launch &L, int fmt, const HitsArgs &a, int T, uint32_t *amax_bits,
                              unsigned long long *counts) {
  size_t nmax = 0;
  for (int t = 0; t < T; ++t) nmax = a.n[t] > nmax ? a.n[t] : nmax;
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, (size_t)T * sizeof(uint32_t), L.stream);
  if (e != cudaSuccess) return e;
  const int grid = stream_grid(L, (nmax + 3) / 4, 1024);
  k_amax_multi_var<<<grid, 256, 0, L.stream>>>(a, T, amax_bits, L.status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (fmt == GIFT_FMT_E4M3) k_hits_multi_var<FMT_E4M3><<<grid, 256, 0, L.stream>>>(a, T, amax_bits, counts);
  else k_hits_multi_var<FMT_E5M2><<<grid, 256, 0, L.stream>>>(a, T, amax_bits, counts);
  return cudaGetLastError();
}

}  // namespace gift
