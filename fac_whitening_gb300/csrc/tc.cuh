// Thin wrappers over the sm_100-family tensor-core PTX used by libgift: tensor memory
// (TMEM) allocation, tcgen05.mma with shared-memory matrix descriptors, tcgen05.commit to an
// mbarrier, and tcgen05.ld of the accumulator.  Hand-written inline PTX (no library).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace gift {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---- TMEM ---------------------------------------------------------------------------------
// One warp allocates `ncols` (power of two >= 32) columns x 128 lanes of 32-bit cells; the
// base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the tensor core's async proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---- mbarrier -----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the barrier phase with a clock budget; false if the budget ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

// ---- MMA ----------------------------------------------------------------------------------
// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 bytes, 8-row
// atoms of 1024 bytes (stride-dimension offset 1024), atom base 1024-byte aligned; the start
// address may be advanced by 32-byte steps inside a row to select the K slice of one MMA.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);      // start address, bits [0,14)
  d |= (uint64_t)1 << 16;                             // leading-dimension offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                   // stride-dimension offset, bits [32,46)
  d |= (uint64_t)1 << 46;                             // descriptor version for this family
  d |= (uint64_t)2 << 61;                             // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: D = F32, A = B = TF32, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor: D = F32, A = B = BF16 (kind::f16), both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 16 BF16 step; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, one 128 x N x 16 BF16 step with A in tensor memory
// (lane m = row m of A, each 32-bit column holds two consecutive K elements, the lower K in the
// low half); issued by one thread.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Registers -> 16 consecutive 32-bit columns of this thread's lane (a warp writes its
// 32-lane slice); tmem_wait_st before the data is used by another agent.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 8 TF32 step; issued by one thread.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Shared memory -> tensor memory: 128 rows x 32 bytes (the K slice a descriptor selects, in
// the operand layouts of the MMA descriptors) into lanes 0-127, 8 consecutive 32-bit columns
// from taddr; asynchronous, in order with this thread's MMAs, tracked by mma_commit.
__device__ __forceinline__ void cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;\n" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ---- TMEM -> registers ----------------------------------------------------------------------
// 32 consecutive 32-bit columns of this thread's lane (a warp reads its 32-lane slice).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r);
__device__ __forceinline__ void tmem_wait_ld(uint32_t *r);
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  tmem_ld32_nowait(taddr, r);
  tmem_wait_ld(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive columns without the completion wait (tmem_wait_ld before using v).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Completion wait for tmem_ld32_nowait; the registers pass through it so that no use of them
// can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 16 consecutive columns without the completion wait, and its wait.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// ---- exact BF16 splitting ------------------------------------------------------------------
// x = t1 + t2 + t3 with each term a BF16 value (round to nearest at every step).  BF16 keeps
// FP32's exponent range, so each remainder is formed exactly (the operands of each
// subtraction are within a factor of two) and 8 + 8 + 8 significant bits cover the 24 of x:
// the last remainder fits in BF16 exactly (values below 2^-110 aside, where BF16 subnormals
// drop bits worth less than 2^-133).
__device__ __forceinline__ void bf16_split3(float x, uint16_t &t1, uint16_t &t2, uint16_t &t3) {
  const __nv_bfloat16 h1 = __float2bfloat16_rn(x);
  const float r1 = __fsub_rn(x, __bfloat162float(h1));
  const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
  const float r2 = __fsub_rn(r1, __bfloat162float(h2));
  const __nv_bfloat16 h3 = __float2bfloat16_rn(r2);
  t1 = __bfloat16_as_ushort(h1);
  t2 = __bfloat16_as_ushort(h2);
  t3 = __bfloat16_as_ushort(h3);
}
// The same split for two values at once, each term pair packed low = x0, high = x1: one
// packed conversion per term instead of two (cvt.rn.bf16x2.f32 puts its first source in the
// upper half), the same roundings and remainders as bf16_split3.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ void bf16_split3x2(float x0, float x1, uint32_t &w1, uint32_t &w2, uint32_t &w3) {
  w1 = pack_bf16x2_rn(x0, x1);
  const float r0 = __fsub_rn(x0, __uint_as_float(w1 << 16)), r1 = __fsub_rn(x1, __uint_as_float(w1 & 0xFFFF0000u));
  w2 = pack_bf16x2_rn(r0, r1);
  const float s0 = __fsub_rn(r0, __uint_as_float(w2 << 16)), s1 = __fsub_rn(r1, __uint_as_float(w2 & 0xFFFF0000u));
  w3 = pack_bf16x2_rn(s0, s1);
}
// Operand planes of the tensor-core apply, for element (row, k < 32) of a rows x 32 operand:
// plane 0 row = [t1 of k = 0..31 | t2 of k = 0..31] (128 bytes), plane 1 row = [t3 | zeros].
// `planes` holds nplanes planes of rows x 64 BF16 each.
__device__ __forceinline__ void write_term_planes(uint16_t *planes, size_t rows, size_t row, int k, float x,
                                                  int nplanes) {
  uint16_t t1, t2, t3;
  bf16_split3(x, t1, t2, t3);
  uint16_t *p0 = planes + row * 64;
  p0[k] = t1;
  p0[32 + k] = t2;
  if (nplanes > 1) {
    uint16_t *p1 = planes + rows * 64 + row * 64;
    p1[k] = t3;
    p1[32 + k] = 0;
  }
}

// The same for 16 consecutive k (kb a multiple of 16), stored as 32-byte runs.
__device__ __forceinline__ void write_term_planes16(uint16_t *planes, size_t rows, size_t row, int kb, const float *x,
                                                    int nplanes) {
  uint32_t w1[8], w2[8], w3[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) bf16_split3x2(x[2 * q], x[2 * q + 1], w1[q], w2[q], w3[q]);
  uint4 *p0 = reinterpret_cast<uint4 *>(planes + row * 64 + kb);
  uint4 *p0b = reinterpret_cast<uint4 *>(planes + row * 64 + 32 + kb);
  p0[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  p0[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
  p0b[0] = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  p0b[1] = make_uint4(w2[4], w2[5], w2[6], w2[7]);
  if (nplanes > 1) {
    uint4 *p1 = reinterpret_cast<uint4 *>(planes + rows * 64 + row * 64 + kb);
    uint4 *p1b = reinterpret_cast<uint4 *>(planes + rows * 64 + row * 64 + 32 + kb);
    p1[0] = make_uint4(w3[0], w3[1], w3[2], w3[3]);
    p1[1] = make_uint4(w3[4], w3[5], w3[6], w3[7]);
    p1b[0] = make_uint4(0u, 0u, 0u, 0u);
    p1b[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---- exact TF32 splitting -----------------------------------------------------------------
// x = t1 + t2 + t3 with each term exactly representable in TF32 (low 13 mantissa bits zero):
// t1 rounds x to 11 significant bits, t2 rounds the exact remainder, t3 is what is left
// (at most 2 significant bits).  All subtractions are exact.
__device__ __forceinline__ float tf32_round(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

}  // namespace tc
}  // namespace gift

namespace gift {
namespace tc {

// ---- TMA (bulk tensor copies) --------------------------------------------------------------
// Expect `bytes` more transaction bytes on `bar` and arrive once.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// 2-D tiled load of the box at element coordinates (x = innermost, y) into shared memory,
// completing `bar`'s transaction count.  x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// bring a tensor map (kernel parameter or global) into the descriptor cache ahead of its use
__device__ __forceinline__ void prefetch_tensormap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(tmap) : "memory");
}
// named barrier for a subset of the CTA's warps
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace tc
}  // namespace gift
