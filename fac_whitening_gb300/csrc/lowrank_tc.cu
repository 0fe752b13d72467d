// Rank-r whitening apply on the 5th-generation tensor cores: a persistent, warp-specialised
// pipeline (TMA loads -> tcgen05.mma into TMEM -> fused read-out).
//
// GIFT reading notes (zhongzhuzhou.org), simplification 2, eq. (17), with the sigma I
// completion: W~ = alpha W + (P diag(c)) U^T with P = W U (see lowrank.cu).  The rank-r
// product Pc U^T (K = 32) is a dense contraction over every element of the tile, so it runs
// on the tensor cores; alpha W, the amax, the FP8/NVFP4 pack or the FP32 store are fused into
// the TMEM read-out.
//
// Operands.  Pc and U are split exactly into three BF16 terms, x = x1 + x2 + x3 (tc.cuh), and
// stored as "term planes": plane 0 row = [x1 | x2] (2 x 32 BF16 = one 128-byte row), plane 1
// row = [x3 | 0].  The FP32 path accumulates the six products x_i y_j with i + j <= 4 (what is
// dropped is below 2^-23 |x||y|, under the rounding of an FP32 dot product of length 32);
// the TC path the three with i + j <= 3 (below 2^-15 |x||y|).  Splitting a wide operand into
// narrow tensor-core terms follows the split-precision idea of H. Ootomo and R. Yokota,
// "Recovering single precision accuracy from Tensor Cores while surpassing the FP32
// theoretical peak performance", IJHPCA 2022.
//
// Tile: 128 rows x 64 columns, D[128 x 64] (FP32, TMEM) = sum over products A_i B_j^T, A = Pc
// rows, B = U rows, K = 32 (two BF16 MMA steps of K = 16 per product).  One CTA per SM; when
// the row blocks are no more than the SMs, each CTA stays inside one row block (its A planes
// are loaded once), otherwise CTAs walk contiguous tile ranges in row-block order.  Warp 8
// issues TMA loads (the W tile as two 128 x 32 boxes and the B planes) into four stages; warp 9
// issues the MMAs into two TMEM accumulators; warps 0-7 read out, two per TMEM lane quarter
// (one tile row and 32 columns per thread).  Full/empty mbarriers connect the roles; every
// wait is clock-bounded and reports GIFT_ERR_TIMEOUT instead of hanging.  The 128-byte TMA
// swizzle gives the tcgen05 K-major operand layout and conflict-free row reads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace gift {

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 64;
constexpr int kBPlane = kTileN * 128;         // 64 rows x 128 bytes
constexpr int kWBox = 128 * 128;              // 128 rows x 32 floats of W
constexpr int kStages = 4;
constexpr int kReadWarps = 8;
constexpr int kThreads = 32 * (kReadWarps + 2);
constexpr uint32_t kTmemCols = 256;           // two 64-column accumulators, then A
constexpr uint32_t kACol = 2 * kTileN;        // A terms: 16 columns each (32 BF16 per lane)
constexpr long long kWaitBudget = 4000000000LL;

struct PipeParams {
  LrApply a;
  int tiles_n, tiles_total;
  int cpr;    // > 0: CTAs per row block (row-aligned schedule); 0: contiguous tile ranges
  int unit;   // tiles handed out together: 2 for the 128 x 128 block epilogues (a block's two
              // 64-column tiles go to one CTA, back to back), else 1
};

template <int NPL>
struct Layout {
  static constexpr int stage_bytes = 2 * kWBox + NPL * kBPlane;
  static constexpr int total = kStages * stage_bytes;
};

__device__ __forceinline__ int sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

}  // namespace

template <int EPI, int F, int NPL, bool TOUT>
__global__ void __launch_bounds__(kThreads, 1) k_lr_apply_pipe(const __grid_constant__ PipeParams P,
                                                               const __grid_constant__ CUtensorMap tmW,
                                                               const __grid_constant__ CUtensorMap tmB, int *status) {
  using Lay = Layout<NPL>;
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_tfull[2], bar_tempty[2];
  __shared__ uint64_t bar_afull, bar_aempty, bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[kReadWarps];
  __shared__ uint32_t redb[2][kReadWarps];   // block amax, double-buffered across blocks
  __shared__ volatile int failed;

  const LrApply &a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = a.d_out, d_in = a.d_in;
  const int b = blockIdx.x;
  int t_begin, t_end;
  const int un = P.unit;
  if (P.cpr > 0) {
    const int rb = b / P.cpr, j = b - rb * P.cpr, units = P.tiles_n / un;
    t_begin = rb * P.tiles_n + un * (int)(((long long)units * j) / P.cpr);
    t_end = rb * P.tiles_n + un * (int)(((long long)units * (j + 1)) / P.cpr);
  } else {
    const int units = P.tiles_total / un;
    t_begin = un * (int)(((long long)units * b) / gridDim.x);
    t_end = un * (int)(((long long)units * (b + 1)) / gridDim.x);
  }

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], kReadWarps);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bar_tfull[s], 1);
      tc::mbar_init(&bar_tempty[s], kReadWarps);
    }
    tc::mbar_init(&bar_afull, kReadWarps);
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

  if (warp == kReadWarps) {
    // ---------------- TMA producer: W tile (two boxes) and the B planes per stage ----------------
    if (lane == 0) {
      int issued[kStages] = {};
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int rb = t / P.tiles_n, cb = t - rb * P.tiles_n;
        const int s = i % kStages;
        if (!wait(&bar_empty[s], ((i / kStages) & 1) ^ 1)) break;
        uint8_t *st = sm + s * Lay::stage_bytes;
        tc::mbar_arrive_expect_tx(&bar_full[s], Lay::stage_bytes);
        tc::tma_load_2d(st, &tmW, cb * kTileN, rb * kTileM, &bar_full[s]);
        tc::tma_load_2d(st + kWBox, &tmW, cb * kTileN + 32, rb * kTileM, &bar_full[s]);
#pragma unroll
        for (int q = 0; q < NPL; ++q)
          tc::tma_load_2d(st + 2 * kWBox + q * kBPlane, &tmB, 0, q * d_in + cb * kTileN, &bar_full[s]);
        ++issued[s];
      }
      if (failed) {
        // bounded drain of the loads still in flight before the CTA's shared memory goes away
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&bar_full[s], (uint32_t)((issued[s] - 1) & 1), kWaitBudget);
      }
    }
  } else if (warp == kReadWarps + 1) {
    // ---------------- MMA issuer: A from TMEM, B from shared memory ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kTileM, kTileN);
      // products x_i y_j (0-based term indices), smallest first: FP32 path i + j <= 2 over
      // three terms, TC path i + j <= 1 over two
      constexpr int np = (NPL == 1) ? 3 : 6;
      constexpr int pa[6] = {NPL == 1 ? 1 : 2, NPL == 1 ? 0 : 1, 0, 1, 0, 0};
      constexpr int pb[6] = {0, 1, NPL == 1 ? 0 : 2, 0, 1, 0};
      int cur_rb = -1;
      uint32_t a_par = 0;
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int rb = t / P.tiles_n;
        const int s = i % kStages, acc_i = i & 1;
        if (rb != cur_rb) {
          if (!wait(&bar_afull, a_par)) break;
          a_par ^= 1;
          cur_rb = rb;
        }
        if (!wait(&bar_full[s], (uint32_t)((i / kStages) & 1))) break;
        if (!wait(&bar_tempty[acc_i], (uint32_t)(((i >> 1) & 1) ^ 1))) break;
        tc::fence_after_sync();
        const uint32_t b0 = tc::smem_u32(sm + s * Lay::stage_bytes + 2 * kWBox);
        uint32_t acc = 0;
#pragma unroll
        for (int p = 0; p < np; ++p) {
          // B term t sits in plane t / 2 at byte offset 64 * (t % 2) of each 128-byte row;
          // A term t in TMEM columns kACol + 16 t (two BF16 per column)
          const uint32_t bb = b0 + (pb[p] >> 1) * kBPlane + 64 * (pb[p] & 1);
#pragma unroll
          for (int k = 0; k < 2; ++k) {   // K = 32 as two steps of 16 BF16
            tc::mma_bf16_ta(tmem + acc_i * kTileN, tmem + kACol + 16 * pa[p] + 8 * k,
                            tc::sdesc_kmajor_sw128(bb + 32 * k), idesc, acc);
            acc = 1;
          }
        }
        tc::mma_commit(&bar_tfull[acc_i]);
        const int nrb = (t + 1 < t_end) ? (t + 1) / P.tiles_n : -1;
        if (nrb != rb) tc::mma_commit(&bar_aempty);   // A of this row block may be replaced
      }
      // every MMA issued has landed in TMEM before the columns are freed
      tc::mma_commit(&bar_done);
      tc::mbar_wait_bounded(&bar_done, 0, kWaitBudget);
    }
  } else {
    // ---------------- read-out (warps 0-7): thread = one tile row, 32 columns ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const int rtid = tid;                          // 0..255
    const double sg = (double)a.sigma[0];
    const float alpha = a.inverse ? (float)sqrt(sg) : (float)(1.0 / sqrt(sg));
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
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
    const int lr = quarter * 32 + lane;            // tile row = TMEM lane
    const uint32_t *pc_planes = reinterpret_cast<const uint32_t *>(a.split);   // rows of 32 words
    int cur_rb = -1;
    uint32_t ae_par = 0;
    // 128 x 128 blocks: the first tile's values (and residual row) wait for the second tile
    float vk[32];
    uint32_t mk = 0;
    float *rk = nullptr;
    int bpar = 0;
    // FP8 codes of 32 values of a row (and, with error feedback, the residual they leave)
    auto pack_fp8_row = [&](const float *vv, const ScalePair &p, uint8_t *dst, float *rdst) {
      uint32_t w4[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float *x = vv + 4 * h;
        w4[h] = pack4_fp8<F>(__fmul_rn(x[0], p.m), __fmul_rn(x[1], p.m), __fmul_rn(x[2], p.m), __fmul_rn(x[3], p.m));
      }
      if (!dst) return;
      uint4 *d4 = reinterpret_cast<uint4 *>(dst);
      d4[0] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      d4[1] = make_uint4(w4[4], w4[5], w4[6], w4[7]);
      if (rdst) {
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          float e[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            e[k] = __fsub_rn(vv[4 * h + k], __fmul_rn(dec_fp8<F>((w4[h] >> (8 * k)) & 0xFFu), p.s));
          reinterpret_cast<float4 *>(rdst)[h] = make_float4(e[0], e[1], e[2], e[3]);
        }
      }
    };
    for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
      const int rb = t / P.tiles_n, cb = t - rb * P.tiles_n;
      const int s = i % kStages, acc_i = i & 1;
      const int r0 = rb * kTileM, c0 = cb * kTileN;
      const int row = r0 + lr;
      if (rb != cur_rb) {
        // A (the Pc term planes of this row block) -> TMEM, once per row block: half 0 writes
        // term 1 (and term 3), half 1 term 2; rows past the matrix edge get zeros
        if (cur_rb >= 0) {
          wait(&bar_aempty, ae_par);
          ae_par ^= 1;
          tc::fence_after_sync();
        }
#pragma unroll
        for (int j = 0; j < ((NPL == 2) ? 2 : 1); ++j) {
          if (half == 1 && j == 1) break;
          const int plane = j, woff = (half == 0) ? 0 : 16;
          const uint32_t col = kACol + (uint32_t)(32 * plane + woff);
          uint32_t r[16];
          if (row < d_out) {
            const uint4 *src = reinterpret_cast<const uint4 *>(pc_planes + ((size_t)plane * d_out + row) * 32 + woff);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 x = src[q];
              r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) r[q] = 0u;
          }
          tc::tmem_st16(tmem + lane_off + col, r);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar_afull);
        cur_rb = rb;
      }
      // after a timeout the read-out still walks its tiles (on whatever the buffers hold, the
      // status already says the output is invalid) so that all eight warps meet the same
      // named barriers; every later wait returns at once
      wait(&bar_tfull[acc_i], (uint32_t)((i >> 1) & 1));
      wait(&bar_full[s], (uint32_t)((i / kStages) & 1));
      tc::fence_after_sync();
      uint32_t raw[32];
      tc::tmem_ld32_nowait(tmem + lane_off + (uint32_t)(acc_i * kTileN + 32 * half), raw);
      uint8_t *st = sm + s * Lay::stage_bytes;
      uint8_t *box = st + half * kWBox;            // this thread's 32 columns of W
      float4 w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const float4 *>(box + sw128(lr, c));
      tc::tmem_wait_ld(raw);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_tempty[acc_i]);

      float v[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        v[4 * c + 0] = fmaf(alpha, w[c].x, __uint_as_float(raw[4 * c + 0]));
        v[4 * c + 1] = fmaf(alpha, w[c].y, __uint_as_float(raw[4 * c + 1]));
        v[4 * c + 2] = fmaf(alpha, w[c].z, __uint_as_float(raw[4 * c + 2]));
        v[4 * c + 3] = fmaf(alpha, w[c].w, __uint_as_float(raw[4 * c + 3]));
      }
      const bool in = row < d_out && (c0 + 32 * half) < d_in;   // d_in is a multiple of 32
      // error feedback: the tensor quantised is U~ = W~ + R
      float *rrow = (a.R && in) ? a.R + (size_t)row * d_in + c0 + 32 * half : nullptr;
      if (rrow) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 r4 = reinterpret_cast<const float4 *>(rrow)[c];
          v[4 * c + 0] = __fadd_rn(v[4 * c + 0], r4.x);
          v[4 * c + 1] = __fadd_rn(v[4 * c + 1], r4.y);
          v[4 * c + 2] = __fadd_rn(v[4 * c + 2], r4.z);
          v[4 * c + 3] = __fadd_rn(v[4 * c + 3], r4.w);
        }
      }
      if (EPI == LR_AMAX && in) {
        // the B planes are stacked in one tensor, so columns past the matrix edge hold
        // neighbouring data: they are kept out of the amax (and never stored)
#pragma unroll
        for (int e = 0; e < 32; ++e) m_run = max(m_run, abs_bits(v[e]));
      }
      if (EPI == LR_STORE || TOUT) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4 *>(box + sw128(lr, c)) = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        tc::named_bar_sync(1, 32 * kReadWarps);
        float *dst = (EPI == LR_STORE) ? a.out : a.tout;
#pragma unroll
        for (int k = 0; k < (kTileM * kTileN / 4) / (32 * kReadWarps); ++k) {
          const int q = k * 32 * kReadWarps + rtid;
          const int rr = q >> 4, c16 = q & 15;
          const int gr = r0 + rr, gc = c0 + 4 * c16;
          if (gr < d_out && gc < d_in)
            *reinterpret_cast<float4 *>(dst + (size_t)gr * d_in + gc) =
                *reinterpret_cast<const float4 *>(st + (c16 >> 3) * kWBox + sw128(rr, c16 & 7));
        }
      }
      if (EPI == LR_PACK_TENSOR)
        pack_fp8_row(v, sp, in ? a.codes + (size_t)row * d_in + c0 + 32 * half : nullptr, rrow);
      if (EPI == LR_BLOCK || EPI == LR_BLOCK_AMAX) {
        // 128 x 128 block scaling (d_in % 128 == 0): the block's amax over both of its tiles,
        // then both tiles packed with the block's scale
        uint32_t mb = 0;
        if (in) {
#pragma unroll
          for (int e = 0; e < 32; ++e) mb = max(mb, abs_bits(v[e]));
        }
        if ((cb & 1) == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e) vk[e] = v[e];
          mk = mb;
          rk = rrow;
        } else {
          mb = warp_max_u32(max(mb, mk));
          if (lane == 0) redb[bpar][warp] = mb;
          tc::named_bar_sync(2, 32 * kReadWarps);
          uint32_t m = 0;
#pragma unroll
          for (int w = 0; w < kReadWarps; ++w) m = max(m, redb[bpar][w]);
          bpar ^= 1;
          const int blk = rb * (d_in / 128) + (cb >> 1);
          if (EPI == LR_BLOCK_AMAX) {
            if (tid == 0) {
              atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws) + blk, m);
              if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
            }
          } else {
            const float bam = a.amax_in ? a.amax_in[blk] : __uint_as_float(m);
            const ScalePair bp = scale_pair(bam, fmax_of<F>());
            if (tid == 0) {
              if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
              reinterpret_cast<float *>(a.scales)[blk] = bp.s;
              if (a.amax_out) a.amax_out[blk] = bam;
            }
            uint8_t *crow = a.codes + (size_t)row * d_in + c0 + 32 * half;
            pack_fp8_row(vk, bp, in ? crow - kTileN : nullptr, rk);
            pack_fp8_row(v, bp, in ? crow : nullptr, rrow);
          }
        }
      }
      if (EPI == LR_NVFP4) {
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
          if (rrow) {   // element e of the group sits in word e / 8, bits 4 (e % 8)
            const float ev = dec_e4m3(grp.e_code);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t word = cw[2 * g + (q >> 1)];
              float e4[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                e4[k] = __fsub_rn(v[16 * g + 4 * q + k], nvfp4_deq((word >> (16 * (q & 1) + 4 * k)) & 0xFu, ev, s_t));
              reinterpret_cast<float4 *>(rrow + 16 * g)[q] = make_float4(e4[0], e4[1], e4[2], e4[3]);
            }
          }
        }
        if (in) {
          *reinterpret_cast<uint4 *>(a.codes + (((size_t)row * d_in + c0 + 32 * half) >> 1)) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(a.scales) + (size_t)row * (d_in / kNvGroup) +
                                        (c0 + 32 * half) / kNvGroup) = sc;
        }
      }
      // this warp's generic-proxy reads (and writes) of the stage are ordered before the
      // async-proxy (TMA) refill
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_empty[s]);
    }
    if (EPI == LR_AMAX) {
      m_run = warp_max_u32(m_run);
      if (lane == 0) red[warp] = m_run;
      tc::named_bar_sync(1, 32 * kReadWarps);
      if (tid == 0) {
        uint32_t m = 0;
        for (int w = 0; w < kReadWarps; ++w) m = max(m, red[w]);
        if (m) atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws), m);
        if (m >= 0x7F800000u) set_status(status, GIFT_ERR_NONFINITE);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// =========================================================================================
// Fused encode: transform, grid-wide amax and pack with W~ held in tensor memory.
//
// Each CTA owns at most kSlots tiles of one row block and keeps every tile's W~ in its own
// 64-column TMEM slot (8 slots = all 512 columns), so W is read from HBM once: phase A runs
// the pipeline above (A = Pc term planes from shared memory, loaded once; B = U planes and W
// streamed per tile), forms W~ = alpha W + Pc U^T, folds it into the CTA amax and writes it
// back into the slot; the CTAs then meet at one grid-wide barrier (launched cooperatively, so
// all CTAs are resident; the wait is clock-bounded) after which every CTA reads the tensor
// amax and packs its tiles straight out of tensor memory (phase B).  With a caller-supplied
// amax there is no barrier.  The arithmetic of W~, the amax and the codes is the same as in
// the two-kernel path (amax pass, then pack pass).
// =========================================================================================
namespace {

constexpr int kSlots = 8;
constexpr int kAPlaneF = 128 * 128;   // Pc plane in shared memory: 128 rows x 128 bytes

struct FusedParams {
  LrApply a;
  int tiles_n;
  int cpr;
  unsigned int *grid_counter;   // zero on entry
};

template <int NPL>
struct FLayout {
  static constexpr int stage_bytes = 2 * kWBox + NPL * kBPlane;
  static constexpr int stage_off = NPL * kAPlaneF;
  static constexpr int total = stage_off + kStages * stage_bytes;
};

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace

template <int EPI, int F, int NPL, bool TOUT>
__global__ void __launch_bounds__(kThreads, 1) k_lr_encode_fused(const __grid_constant__ FusedParams P,
                                                                 const __grid_constant__ CUtensorMap tmW,
                                                                 const __grid_constant__ CUtensorMap tmA,
                                                                 const __grid_constant__ CUtensorMap tmB, int *status) {
  using Lay = FLayout<NPL>;
  extern __shared__ uint8_t dsm[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_tfull[kSlots], bar_afull;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t red[kReadWarps];
  __shared__ float amax_sh;
  __shared__ volatile int failed;

  const LrApply &a = P.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d_out = a.d_out, d_in = a.d_in;
  const int b = blockIdx.x;
  const int rb = b / P.cpr, jc = b - rb * P.cpr;
  const int t_begin = rb * P.tiles_n + (int)(((long long)P.tiles_n * jc) / P.cpr);
  const int t_end = rb * P.tiles_n + (int)(((long long)P.tiles_n * (jc + 1)) / P.cpr);
  const int r0 = rb * kTileM;

  if (warp == 0) {
    tc::tmem_alloc(&tmem_base_sh, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], kReadWarps);
    }
    for (int s = 0; s < kSlots; ++s) tc::mbar_init(&bar_tfull[s], 1);
    tc::mbar_init(&bar_afull, 1);
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

  if (warp == kReadWarps) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued[kStages] = {};
      bool a_issued = false;
      if (t_end > t_begin) {
        tc::mbar_arrive_expect_tx(&bar_afull, NPL * kAPlaneF);
#pragma unroll
        for (int q = 0; q < NPL; ++q) tc::tma_load_2d(sm + q * kAPlaneF, &tmA, 0, q * d_out + r0, &bar_afull);
        a_issued = true;
      }
      for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
        const int cb = t - rb * P.tiles_n;
        const int s = i % kStages;
        if (!wait(&bar_empty[s], ((i / kStages) & 1) ^ 1)) break;
        uint8_t *st = sm + Lay::stage_off + s * Lay::stage_bytes;
        tc::mbar_arrive_expect_tx(&bar_full[s], Lay::stage_bytes);
        tc::tma_load_2d(st, &tmW, cb * kTileN, r0, &bar_full[s]);
        tc::tma_load_2d(st + kWBox, &tmW, cb * kTileN + 32, r0, &bar_full[s]);
#pragma unroll
        for (int q = 0; q < NPL; ++q)
          tc::tma_load_2d(st + 2 * kWBox + q * kBPlane, &tmB, 0, q * d_in + cb * kTileN, &bar_full[s]);
        ++issued[s];
      }
      if (failed) {
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) tc::mbar_wait_bounded(&bar_full[s], (uint32_t)((issued[s] - 1) & 1), kWaitBudget);
        if (a_issued) tc::mbar_wait_bounded(&bar_afull, 0, kWaitBudget);
      }
    }
  } else if (warp == kReadWarps + 1) {
    // ---------------- MMA issuer: one TMEM slot per tile ----------------
    if (lane == 0 && t_end > t_begin) {
      constexpr uint32_t idesc = tc::idesc_bf16(kTileM, kTileN);
      constexpr int np = (NPL == 1) ? 3 : 6;
      constexpr int pa[6] = {NPL == 1 ? 1 : 2, NPL == 1 ? 0 : 1, 0, 1, 0, 0};
      constexpr int pb[6] = {0, 1, NPL == 1 ? 0 : 2, 0, 1, 0};
      if (wait(&bar_afull, 0)) {
        const uint32_t a0 = tc::smem_u32(sm);
        for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
          const int s = i % kStages;
          if (!wait(&bar_full[s], (uint32_t)((i / kStages) & 1))) break;
          tc::fence_after_sync();
          const uint32_t b0 = tc::smem_u32(sm + Lay::stage_off + s * Lay::stage_bytes + 2 * kWBox);
          uint32_t acc = 0;
#pragma unroll
          for (int p = 0; p < np; ++p) {
            const uint32_t aa = a0 + (pa[p] >> 1) * kAPlaneF + 64 * (pa[p] & 1);
            const uint32_t bb = b0 + (pb[p] >> 1) * kBPlane + 64 * (pb[p] & 1);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              tc::mma_bf16(tmem + (uint32_t)(i * kTileN), tc::sdesc_kmajor_sw128(aa + 32 * k),
                           tc::sdesc_kmajor_sw128(bb + 32 * k), idesc, acc);
              acc = 1;
            }
          }
          tc::mma_commit(&bar_tfull[i]);
        }
      }
    }
  } else {
    // ---------------- read-out (warps 0-7): thread = one tile row, 32 columns ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const double sg = (double)a.sigma[0];
    const float alpha = a.inverse ? (float)sqrt(sg) : (float)(1.0 / sqrt(sg));
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int lr = quarter * 32 + lane;
    const int row = r0 + lr;
    uint32_t m_run = 0;
    // phase A: W~ of every tile into its slot, CTA amax
    for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
      const int cb = t - rb * P.tiles_n, c0 = cb * kTileN;
      const int s = i % kStages;
      wait(&bar_tfull[i], 0);
      wait(&bar_full[s], (uint32_t)((i / kStages) & 1));
      tc::fence_after_sync();
      const uint32_t slot = tmem + lane_off + (uint32_t)(i * kTileN + 32 * half);
      uint32_t raw[32];
      tc::tmem_ld32_nowait(slot, raw);
      const uint8_t *box = sm + Lay::stage_off + s * Lay::stage_bytes + half * kWBox;
      float4 w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const float4 *>(box + sw128(lr, c));
      tc::tmem_wait_ld(raw);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        raw[4 * c + 0] = __float_as_uint(fmaf(alpha, w[c].x, __uint_as_float(raw[4 * c + 0])));
        raw[4 * c + 1] = __float_as_uint(fmaf(alpha, w[c].y, __uint_as_float(raw[4 * c + 1])));
        raw[4 * c + 2] = __float_as_uint(fmaf(alpha, w[c].z, __uint_as_float(raw[4 * c + 2])));
        raw[4 * c + 3] = __float_as_uint(fmaf(alpha, w[c].w, __uint_as_float(raw[4 * c + 3])));
      }
      // W was read through the generic proxy and the refill writes through the async (TMA)
      // proxy: order the reads before the hand-back
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_empty[s]);
      const bool in = row < d_out && (c0 + 32 * half) < d_in;
      if (in) {
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
      tc::tmem_st16(slot, raw);
      tc::tmem_st16(slot + 16, raw + 16);
      tc::tmem_wait_st();
    }
    // CTA amax, then (without a caller amax) the grid-wide maximum
    m_run = warp_max_u32(m_run);
    if (lane == 0) red[warp] = m_run;
    tc::named_bar_sync(1, 32 * kReadWarps);
    if (tid == 0) {
      uint32_t m = 0;
      for (int w = 0; w < kReadWarps; ++w) m = max(m, red[w]);
      float amax;
      if (a.amax_in) {
        amax = a.amax_in[0];
      } else {
        if (m) atomicMax(reinterpret_cast<uint32_t *>(a.amax_ws), m);
        __threadfence();
        atomicAdd(P.grid_counter, 1u);
        const long long t0 = clock64();
        while (ld_acquire_u32(P.grid_counter) < gridDim.x) {
          if (clock64() - t0 > kWaitBudget) {
            set_status(status, GIFT_ERR_TIMEOUT);
            break;
          }
          __nanosleep(64);
        }
        amax = __uint_as_float(ld_acquire_u32(reinterpret_cast<const unsigned int *>(a.amax_ws)));
      }
      amax_sh = amax;
      if (b == 0) {
        if (!(amax <= kF32Max)) set_status(status, GIFT_ERR_NONFINITE);
        if (EPI == LR_PACK_TENSOR) reinterpret_cast<float *>(a.scales)[0] = scale_pair(amax, fmax_of<F>()).s;
        else a.tscale[0] = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
        if (a.amax_out) a.amax_out[0] = amax;
      }
    }
    tc::named_bar_sync(1, 32 * kReadWarps);
    const float amax = amax_sh;
    const ScalePair sp = scale_pair(amax, fmax_of<F>());
    const float s_t = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, kNvfp4TensorDiv);
    // phase B: pack every tile out of its slot
    for (int t = t_begin, i = 0; t < t_end; ++t, ++i) {
      const int cb = t - rb * P.tiles_n, c0 = cb * kTileN;
      uint32_t raw[32];
      tc::tmem_ld32_nowait(tmem + lane_off + (uint32_t)(i * kTileN + 32 * half), raw);
      tc::tmem_wait_ld(raw);
      float v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(raw[e]);
      const bool in = row < d_out && (c0 + 32 * half) < d_in;
      if (EPI == LR_PACK_TENSOR) {
        uint32_t w4[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float *x = v + 4 * h;
          w4[h] = pack4_fp8<F>(__fmul_rn(x[0], sp.m), __fmul_rn(x[1], sp.m), __fmul_rn(x[2], sp.m),
                               __fmul_rn(x[3], sp.m));
        }
        if (in) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.codes + (size_t)row * d_in + c0 + 32 * half);
          dst[0] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          dst[1] = make_uint4(w4[4], w4[5], w4[6], w4[7]);
        }
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
        if (in) {
          *reinterpret_cast<uint4 *>(a.codes + (((size_t)row * d_in + c0 + 32 * half) >> 1)) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(a.scales) + (size_t)row * (d_in / kNvGroup) +
                                        (c0 + 32 * half) / kNvGroup) = sc;
        }
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

// =========================================================================================
// BF16 term planes of a rows x ld matrix (first kvalid columns, zero beyond, 32 in all)
// =========================================================================================
__global__ void k_split_planes(const float *__restrict__ src, int rows, int ld, int kvalid, int nplanes,
                               uint16_t *__restrict__ dst) {
  const size_t n = (size_t)rows * 32;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const size_t r = i >> 5;
    const int k = (int)(i & 31);
    const float x = (k < kvalid) ? src[r * ld + k] : 0.0f;
    tc::write_term_planes(dst, (size_t)rows, r, k, x, nplanes);
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

// Tensor-core workspace: Pc planes, U planes (the apply), U^T planes (the projection) and the
// projection's row-block counters (see kernels.cuh).
size_t lr_pipe_split_floats(int d_out, int d_in) {
  const size_t blocks = ((size_t)d_out + 127) / 128;
  return (size_t)64 * ((size_t)d_out + d_in) + (size_t)48 * d_in + ((blocks + 63) / 64) * 64;
}

// The pipelined apply covers the per-tensor FP8, NVFP4, amax and store epilogues with
// d_in % 32 == 0 (TMA boxes of 32 columns, 16-byte aligned rows) and the 128 x 128 block FP8
// and block amax epilogues with d_in % 128 == 0, with or without a residual, for 16-byte
// aligned tensors, rank <= 32 and a term-plane workspace; other cases use the FP32-SIMT
// apply in lowrank.cu.
bool lr_apply_tc_ok(const LrApply &a, int epi) {
  const bool block = (epi == LR_BLOCK || epi == LR_BLOCK_AMAX);
  if (epi != LR_AMAX && epi != LR_PACK_TENSOR && epi != LR_NVFP4 && epi != LR_STORE && !block) return false;
  if (!a.split || !a.u_planes) return false;
  if (block && a.d_in % 128 != 0) return false;
  bool ok = (a.d_in % 32 == 0) && aligned16(a.X) && aligned16(a.split) && aligned16(a.u_planes) &&
            (!a.R || aligned16(a.R)) && (!a.tout || aligned16(a.tout)) && a.rank >= 1 && a.rank <= 32;
  if (epi == LR_STORE) ok = ok && aligned16(a.out);
  if (epi == LR_PACK_TENSOR || epi == LR_NVFP4 || epi == LR_BLOCK) ok = ok && aligned16(a.codes);
  if (epi == LR_NVFP4) ok = ok && ((uintptr_t)a.scales & 1) == 0;   // two scale bytes per store
  return ok && tensor_map_encoder() != nullptr;
}

static int pipe_planes(const LrApply &a) { return a.terms == 1 ? 1 : 2; }

// U planes go after the Pc planes (which the finalize writes) in the workspace.
cudaError_t launch_lr_split_u(const Launch &L, const LrApply &a) {
  uint16_t *uplanes = reinterpret_cast<uint16_t *>(a.split + (size_t)2 * 32 * a.d_out);   // workspace planes
  const size_t n = (size_t)a.d_in * 32;
  int grid = (int)((n + 255) / 256);
  if (grid > L.sms * 8) grid = L.sms * 8;
  k_split_planes<<<grid, 256, 0, L.stream>>>(a.U, a.d_in, a.rank, a.rank, pipe_planes(a), uplanes);
  return cudaGetLastError();
}

template <int EPI, int F, int NPL>
static cudaError_t pipe_launch(const Launch &L, const LrApply &a) {
  CUtensorMap tmW, tmB;
  const void *ut = a.u_planes;
  // the U planes are 128-byte rows, mapped as 32 FP32 "columns" (TMA copies bytes)
  if (!make_map(&tmW, a.X, (uint64_t)a.d_out, (uint64_t)a.d_in, kTileM) ||
      !make_map(&tmB, ut, (uint64_t)NPL * a.d_in, 32, kTileN))
    return cudaErrorInvalidValue;
  PipeParams P;
  P.a = a;
  P.tiles_n = (a.d_in + kTileN - 1) / kTileN;
  P.unit = (EPI == LR_BLOCK || EPI == LR_BLOCK_AMAX) ? 2 : 1;
  const int tiles_m = (a.d_out + kTileM - 1) / kTileM;
  P.tiles_total = P.tiles_n * tiles_m;
  int grid;
  if (tiles_m <= L.sms) {
    // row-aligned: every CTA stays in one row block, so A is loaded once per CTA
    P.cpr = L.sms / tiles_m;
    if (P.cpr > P.tiles_n / P.unit) P.cpr = P.tiles_n / P.unit;
    grid = tiles_m * P.cpr;
  } else {
    P.cpr = 0;
    grid = L.sms;
  }
  const int smem = Layout<NPL>::total + 1024;
  cudaError_t e;
  if (a.tout) {
    if ((e = ensure_dynamic_smem<k_lr_apply_pipe<EPI, F, NPL, true>>(smem)) != cudaSuccess) return e;
    k_lr_apply_pipe<EPI, F, NPL, true><<<grid, kThreads, smem, L.stream>>>(P, tmW, tmB, L.status);
  } else {
    if ((e = ensure_dynamic_smem<k_lr_apply_pipe<EPI, F, NPL, false>>(smem)) != cudaSuccess) return e;
    k_lr_apply_pipe<EPI, F, NPL, false><<<grid, kThreads, smem, L.stream>>>(P, tmW, tmB, L.status);
  }
  return cudaGetLastError();
}

template <int NPL>
static cudaError_t pipe_dispatch(const Launch &L, int epi, int fmt, const LrApply &a) {
  switch (epi) {
    case LR_AMAX: return pipe_launch<LR_AMAX, FMT_E4M3, NPL>(L, a);
    case LR_STORE: return pipe_launch<LR_STORE, FMT_E4M3, NPL>(L, a);
    case LR_NVFP4: return pipe_launch<LR_NVFP4, FMT_E4M3, NPL>(L, a);
    case LR_PACK_TENSOR:
      return fmt == GIFT_FMT_E5M2 ? pipe_launch<LR_PACK_TENSOR, FMT_E5M2, NPL>(L, a)
                                  : pipe_launch<LR_PACK_TENSOR, FMT_E4M3, NPL>(L, a);
    case LR_BLOCK_AMAX: return pipe_launch<LR_BLOCK_AMAX, FMT_E4M3, NPL>(L, a);
    case LR_BLOCK:
      return fmt == GIFT_FMT_E5M2 ? pipe_launch<LR_BLOCK, FMT_E5M2, NPL>(L, a)
                                  : pipe_launch<LR_BLOCK, FMT_E4M3, NPL>(L, a);
  }
  return cudaErrorInvalidValue;
}

// Fused encode plan: CTAs per row block so that no CTA has more than kSlots tiles, all CTAs
// resident at once (one per SM).  Returns the grid size, 0 if the shape does not fit.
static int fused_plan(const Launch &L, const LrApply &a, int *cpr_out) {
  const int tiles_n = (a.d_in + kTileN - 1) / kTileN;
  const int tiles_m = (a.d_out + kTileM - 1) / kTileM;
  if (tiles_m > L.sms) return 0;
  int cpr = (tiles_n + kSlots - 1) / kSlots;
  const int spread = L.sms / tiles_m;
  if (spread > cpr) cpr = spread < tiles_n ? spread : tiles_n;
  if ((long long)cpr * tiles_m > L.sms) return 0;
  *cpr_out = cpr;
  return cpr * tiles_m;
}

bool lr_encode_fused_ok(const Launch &L, const LrApply &a, int epi) {
  if (epi != LR_PACK_TENSOR && epi != LR_NVFP4) return false;
  if (!lr_apply_tc_ok(a, epi) || !a.grid_counter || a.R) return false;
  int cpr = 0;
  return fused_plan(L, a, &cpr) > 0;
}

template <int EPI, int F, int NPL, bool TOUT>
static cudaError_t fused_launch(const Launch &L, const LrApply &a, int grid, int cpr) {
  CUtensorMap tmW, tmA, tmB;
  const float *pc = a.split;
  const void *ut = a.u_planes;
  if (!make_map(&tmW, a.X, (uint64_t)a.d_out, (uint64_t)a.d_in, kTileM) ||
      !make_map(&tmA, pc, (uint64_t)NPL * a.d_out, 32, kTileM) ||
      !make_map(&tmB, ut, (uint64_t)NPL * a.d_in, 32, kTileN))
    return cudaErrorInvalidValue;
  FusedParams P;
  P.a = a;
  P.tiles_n = (a.d_in + kTileN - 1) / kTileN;
  P.cpr = cpr;
  P.grid_counter = a.grid_counter;
  const int smem = FLayout<NPL>::total + 1024;
  auto kern = k_lr_encode_fused<EPI, F, NPL, TOUT>;
  cudaError_t e;
  if ((e = ensure_dynamic_smem<k_lr_encode_fused<EPI, F, NPL, TOUT>>(smem)) != cudaSuccess) return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return e;
  if (per_sm < 1 || grid > per_sm * L.sms) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P, tmW, tmA, tmB, L.status);
}

template <int NPL>
static cudaError_t fused_dispatch(const Launch &L, int epi, int fmt, const LrApply &a, int grid, int cpr) {
  if (epi == LR_NVFP4)
    return a.tout ? fused_launch<LR_NVFP4, FMT_E4M3, NPL, true>(L, a, grid, cpr)
                  : fused_launch<LR_NVFP4, FMT_E4M3, NPL, false>(L, a, grid, cpr);
  if (fmt == GIFT_FMT_E5M2)
    return a.tout ? fused_launch<LR_PACK_TENSOR, FMT_E5M2, NPL, true>(L, a, grid, cpr)
                  : fused_launch<LR_PACK_TENSOR, FMT_E5M2, NPL, false>(L, a, grid, cpr);
  return a.tout ? fused_launch<LR_PACK_TENSOR, FMT_E4M3, NPL, true>(L, a, grid, cpr)
                : fused_launch<LR_PACK_TENSOR, FMT_E4M3, NPL, false>(L, a, grid, cpr);
}

// The caller has zeroed a.amax_ws (without a caller amax) and a.grid_counter on L.stream.
cudaError_t launch_lr_encode_fused(const Launch &L, int epi, int fmt, const LrApply &a) {
  int cpr = 0;
  const int grid = fused_plan(L, a, &cpr);
  if (grid <= 0) return cudaErrorInvalidValue;
  return a.terms == 1 ? fused_dispatch<1>(L, epi, fmt, a, grid, cpr) : fused_dispatch<2>(L, epi, fmt, a, grid, cpr);
}

cudaError_t launch_lr_apply_tc(const Launch &L, int epi, int fmt, const LrApply &a, bool single_term) {
  return single_term ? pipe_dispatch<1>(L, epi, fmt, a) : pipe_dispatch<2>(L, epi, fmt, a);
}

}  // namespace gift
