// C ABI of libgift: argument validation, workspace layout and kernel sequencing.
//
// Each entry point validates its arguments on the host, carves the caller's workspace
// with the same layout function that gift_workspace_bytes uses, and enqueues kernels on
// the caller's stream.  No call allocates or frees device memory and no call synchronises.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <vector>

#include "kernels.cuh"

using namespace gift;

namespace {

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

constexpr size_t kAlign = 256;

// Bump allocator over the caller's workspace; with base == nullptr it only measures.
struct Carve {
  char *base;
  size_t off = 0;
  explicit Carve(void *b) : base(static_cast<char *>(b)) {}
  template <typename T>
  T *take(size_t count) {
    off = (off + kAlign - 1) / kAlign * kAlign;
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

bool valid_fmt(gift_format f) { return f >= GIFT_FMT_F32 && f <= GIFT_FMT_NVFP4; }
bool valid_scaling(gift_scaling s) {
  return s == GIFT_SCALE_TENSOR || s == GIFT_SCALE_BLOCK128 || s == GIFT_SCALE_BLOCK512;
}
bool valid_kind(gift_xform k) { return k >= GIFT_XF_IDENTITY && k <= GIFT_XF_CHOL_TWO_SIDED; }

// ---- codec workspace (encode / amax / decode) -----------------------------------------
struct CodecWs {
  float *amax = nullptr;   // amax word at [0], grid-barrier word at [16] (64 floats reserved)
  float *part = nullptr;   // LOWRANK: nsplit x d_out x 32 slice partials of X U
  float *Pc = nullptr;     // LOWRANK: d_out x 32
  float *xbuf = nullptr;   // transformed tensor (CHOL encode) or dequantised input (decode)
  float *tbuf = nullptr;   // CHOL_TWO_SIDED intermediate
  float *split = nullptr;  // LOWRANK: tensor-core operand planes and counters (kernels.cuh)
  float *bpart = nullptr;  // LOWRANK, batched encode: kBatchWs x lr_batch_part_floats
  uint16_t *bplanes = nullptr;   // LOWRANK, batched encode: kBatchWs x 2 x d_out rows of 64 BF16
  float *rdavg = nullptr;        // reduce and decode: the average, after the decode's workspace
  void *gplanes = nullptr;       // CHOL: BF16 term planes of the tensor-core GEMMs' operands
  int nsplit = 0;
  size_t bytes = 0;
};

CodecWs codec_layout(void *base, int sms, gift_op op, gift_xform kind, int d_out, int d_in) {
  CodecWs w;
  Carve c(base);
  const size_t n = (size_t)d_out * d_in;
  w.amax = c.take<float>(64);
  if (kind == GIFT_XF_LOWRANK) {
    w.nsplit = lr_proj_splits(sms, d_out, d_in);
    w.part = c.take<float>(lr_part_floats(sms, d_out, d_in));
    w.Pc = c.take<float>((size_t)d_out * 32);
    w.split = c.take<float>(lr_pipe_split_floats(d_out, d_in));
    const size_t bp = lr_batch_part_floats(sms, d_out, d_in);
    if (bp && (op == GIFT_OP_ENCODE || op == GIFT_OP_AMAX)) {
      w.bpart = c.take<float>((size_t)kBatchWs * bp);
      w.bplanes = c.take<uint16_t>((size_t)kBatchWs * 2 * d_out * 64);
    }
  }
  const bool rd = (op == GIFT_OP_REDUCE_DECODE);
  if (rd) op = GIFT_OP_DECODE;   // the decode's workspace, then the average
  if (kind != GIFT_XF_IDENTITY) {
    if (op == GIFT_OP_DECODE || kind == GIFT_XF_CHOL_INPUT || kind == GIFT_XF_CHOL_TWO_SIDED)
      w.xbuf = c.take<float>(n);
    if (kind == GIFT_XF_CHOL_TWO_SIDED) w.tbuf = c.take<float>(n);
    if (kind == GIFT_XF_CHOL_INPUT || kind == GIFT_XF_CHOL_TWO_SIDED) {
      // X L^-T (or X L^T) has K = d_in; the left factor's product K = d_out
      size_t g = gemm_tc_ws_bytes(d_out, d_in, d_in, 3);
      if (kind == GIFT_XF_CHOL_TWO_SIDED) g = std::max(g, gemm_tc_ws_bytes(d_out, d_in, d_out, 3));
      w.gplanes = c.take<uint8_t>(g);
    }
  }
  if (rd && kind != GIFT_XF_IDENTITY) w.rdavg = c.take<float>(n);
  w.bytes = c.off;
  return w;
}

// ---- factor-update workspace -------------------------------------------------------------
struct FactorWs {
  float *A = nullptr;       // d_in x d_in
  // LOWRANK
  int k = 0, gsplits = 1, ysplits = 1;
  float *Y = nullptr, *Q = nullptr, *yparts = nullptr;
  double *Q64 = nullptr, *Gp = nullptr, *G = nullptr, *Rinv = nullptr, *V = nullptr, *ev = nullptr, *tr = nullptr;
  double *sq = nullptr;     // per-CTA partial sums of a^2
  // CHOL
  double *A64 = nullptr, *Ai64 = nullptr, *work = nullptr;
  float *Gf = nullptr;
  double *G64 = nullptr, *Gi64 = nullptr;
  void *at = nullptr;       // BF16 transpose of the activations (tensor-core SYRK), or the
                            // activations' BF16 term planes (tensor-core FP32 SYRK)
  size_t at_bytes = 0;
  // LOWRANK on the tensor cores (FP32 refresh)
  uint16_t *apl = nullptr, *qpl = nullptr;   // term planes of A (explicit sketch) and of Q^T
  uint16_t *xpl = nullptr, *zpl = nullptr;   // term planes of FP32 activations (T rows) and of Z^T
  float *Z = nullptr;                        // Z = a Q, T x 64
  float *parts = nullptr;                    // split-K partials of A Q or a^T Z
  int ksplit = 1;
  bool implicit = true;
  float *B32 = nullptr, *V32 = nullptr, *th = nullptr, *G32 = nullptr, *R32 = nullptr;
  float *gparts = nullptr, *rparts = nullptr;
  int *flag = nullptr;
  size_t bytes = 0;
};

// Bytes of the activations' BF16 term planes for the tensor-core K-FAC product: rows padded to
// 128, T to 64; three planes cover FP32 activations, BF16 ones need one.
size_t syrk_planes_bytes(int d, int T) {
  const size_t rows = (size_t)(d + 127) / 128 * 128, ldk = (size_t)(T + 63) / 64 * 64;
  return 3 * rows * ldk * 2;
}

FactorWs factor_layout(void *base, int sms, gift_xform kind, int d_out, int d_in, int T, bool implicit = true) {
  FactorWs w;
  Carve c(base);
  w.A = c.take<float>((size_t)d_in * d_in);
  if (T > 0) {
    const int dmax = (kind == GIFT_XF_CHOL_TWO_SIDED && d_out > d_in) ? d_out : d_in;
    w.at_bytes = std::max(syrk_tc_scratch_bytes(dmax, T), syrk_planes_bytes(dmax, T));
    w.at = c.take<uint8_t>(w.at_bytes);
  }
  if (kind == GIFT_XF_LOWRANK) {
    w.k = d_in < 64 ? d_in : 64;
    w.gsplits = d_in / 64;   // the FP64 Gram slices: up to one CTA per SM
    if (w.gsplits < 1) w.gsplits = 1;
    if (w.gsplits > sms) w.gsplits = sms;
    const int rowtiles = (d_in + 127) / 128;
    w.ysplits = (2 * sms + rowtiles - 1) / rowtiles;
    const int maxs = (d_in + 255) / 256;
    if (w.ysplits > maxs) w.ysplits = maxs;
    if (w.ysplits < 1) w.ysplits = 1;
    const size_t dk = (size_t)d_in * w.k;
    w.Y = c.take<float>(dk);
    w.Q = c.take<float>(dk);
    w.yparts = c.take<float>(sgemm_splitk_parts(d_in, w.k, w.ysplits));
    w.Q64 = c.take<double>(dk);
    w.Gp = c.take<double>((size_t)w.gsplits * w.k * w.k);
    w.G = c.take<double>(64 * 64);
    w.Rinv = c.take<double>(64 * 64);
    w.V = c.take<double>(64 * 64);
    w.ev = c.take<double>(64);
    w.tr = c.take<double>(1);
    w.sq = c.take<double>((size_t)trace_partials(sms));
    if (w.k == 64 && d_in > 64) {
      // T == 0: the factor of a given A (explicit sketch, no activations)
      const size_t rows = (size_t)(d_in + 127) / 128 * 128, ldk = (size_t)(d_in + 63) / 64 * 64;
      const size_t rows_t = (size_t)(T + 127) / 128 * 128, ldt = (size_t)(T + 63) / 64 * 64;
      w.implicit = implicit && T > 0;
      if (!w.implicit) w.apl = c.take<uint16_t>(3 * rows * ldk);
      w.qpl = c.take<uint16_t>(3 * 128 * ldk);
      if (T > 0) {
        w.xpl = c.take<uint16_t>(3 * rows_t * ldk);   // the activations as term planes
        w.zpl = c.take<uint16_t>(3 * 128 * ldt);
        w.Z = c.take<float>((size_t)T * 64);
      }
      // split-K of the d-row products (A Q over K = d, or a^T Z over K = T)
      const int tiles_m = (int)(rows / 128), nch = (int)((w.implicit ? ldt : ldk) / 64);
      w.ksplit = std::max(1, std::min(sms / tiles_m, nch));
      w.parts = c.take<float>(gemm_tc_parts_floats(d_in, 64, w.ksplit));
      w.B32 = c.take<float>(64 * 64);
      w.V32 = c.take<float>(64 * 64);
      w.G32 = c.take<float>(64 * 64);
      w.R32 = c.take<float>(64 * 64);
      w.th = c.take<float>(64);
      w.gparts = c.take<float>((size_t)refresh_gram_ctas(sms, std::max(d_in, T)) * 64 * 64);
      w.rparts = c.take<float>((size_t)ritz_rotate_ctas(sms, d_in) * 64);
      w.flag = c.take<int>(1);
    }
  } else if (kind == GIFT_XF_CHOL_INPUT || kind == GIFT_XF_CHOL_TWO_SIDED) {
    const int nmax = d_in > d_out ? d_in : d_out;
    w.A64 = c.take<double>((size_t)d_in * d_in);
    w.Ai64 = c.take<double>((size_t)d_in * d_in);
    w.work = c.take<double>(chol_inv_work_doubles(nmax));
    if (kind == GIFT_XF_CHOL_TWO_SIDED) {
      w.Gf = c.take<float>((size_t)d_out * d_out);
      w.G64 = c.take<double>((size_t)d_out * d_out);
      w.Gi64 = c.take<double>((size_t)d_out * d_out);
    }
  }
  w.bytes = c.off;
  return w;
}

#define CK(expr)                      \
  do {                                \
    const cudaError_t ck_e_ = (expr); \
    if (ck_e_ != cudaSuccess) {       \
      record_cuda_error(ck_e_);       \
      return GIFT_ERR_CUDA;           \
    }                                 \
  } while (0)

Launch mk(const gift_ctx *ctx, int *st, cudaStream_t s) {
  Launch L;
  L.stream = s;
  L.sms = ctx->sms;
  L.status = st;
  L.barrier_wait = ctx->barrier_wait;
  return L;
}

gift_status check_factor(const gift_factor *f, int d_out, int d_in) {
  if (!f || f->kind == GIFT_XF_IDENTITY) return GIFT_OK;
  if (!valid_kind(f->kind)) return GIFT_ERR_INVALID_ARG;
  if (f->d_in != d_in || f->d_out != d_out) return GIFT_ERR_INVALID_ARG;
  if (f->kind == GIFT_XF_LOWRANK) {
    if (!f->U || !f->mu || !f->sigma) return GIFT_ERR_INVALID_ARG;
    if (f->rank < 1 || f->rank > kMaxRank || f->rank > d_in) return GIFT_ERR_INVALID_ARG;
    if (f->planes && !aligned16(f->planes)) return GIFT_ERR_INVALID_ARG;
  } else {
    if (!f->LA || !f->LAinv) return GIFT_ERR_INVALID_ARG;
    if (f->kind == GIFT_XF_CHOL_TWO_SIDED && (!f->LG || !f->LGinv)) return GIFT_ERR_INVALID_ARG;
  }
  return GIFT_OK;
}

gift_xform kind_of(const gift_factor *f) { return f ? f->kind : GIFT_XF_IDENTITY; }

// One product of a full-rank transform: on the tensor cores with exact BF16 operand splits
// (three terms and six products at FP32 precision, two terms and three products at TC
// precision), or FP32 SIMT where the tensor-core path does not apply.
cudaError_t chol_gemm(const Launch &L, const GemmArgs &g, const CodecWs &w, gift_precision prec) {
  if (gemm_tc_ok(g, w.gplanes)) return launch_gemm_tc(L, g, prec == GIFT_PREC_TC ? 2 : 3, w.gplanes);
  return launch_sgemm(L, g);
}

// Full-rank transforms as GEMMs with the explicit inverses of the factor: W~ = L_G^-1 W L_A^-T
// ([notes] core idea step 3, eq. (11)) or W L_A^-T (simplification 1, eq. (16)).  The two-sided
// form takes W L_A^-T first, then L_G^-1 of it.
cudaError_t chol_whiten(const Launch &L, const gift_factor *f, const float *W, int d_out, int d_in,
                        const CodecWs &w, gift_precision prec) {
  const bool two = f->kind == GIFT_XF_CHOL_TWO_SIDED;
  GemmArgs g{};
  g.A = W; g.B = f->LAinv; g.C = two ? w.tbuf : w.xbuf;
  g.M = d_out; g.N = d_in; g.K = d_in; g.lda = d_in; g.ldb = d_in; g.ldc = d_in;
  g.transB = true; g.b_lower_t = true; g.alpha = 1.0f;
  cudaError_t e = chol_gemm(L, g, w, prec);
  if (e != cudaSuccess || !two) return e;
  GemmArgs h{};
  h.A = f->LGinv; h.B = w.tbuf; h.C = w.xbuf;
  h.M = d_out; h.N = d_in; h.K = d_out; h.lda = d_out; h.ldb = d_in; h.ldc = d_in;
  h.a_lower = true; h.alpha = 1.0f;
  return chol_gemm(L, h, w, prec);
}

// The map back ([notes] eq. (14)): W^ = L_G X L_A^T, or X L_A^T for the input side only.
cudaError_t chol_unwhiten(const Launch &L, const gift_factor *f, const float *X, int d_out, int d_in, float *out,
                          const CodecWs &w, gift_precision prec) {
  const bool two = f->kind == GIFT_XF_CHOL_TWO_SIDED;
  GemmArgs g{};
  g.A = X; g.B = f->LA; g.C = two ? w.tbuf : out;
  g.M = d_out; g.N = d_in; g.K = d_in; g.lda = d_in; g.ldb = d_in; g.ldc = d_in;
  g.transB = true; g.b_lower_t = true; g.alpha = 1.0f;
  cudaError_t e = chol_gemm(L, g, w, prec);
  if (e != cudaSuccess || !two) return e;
  GemmArgs h{};
  h.A = f->LG; h.B = w.tbuf; h.C = out;
  h.M = d_out; h.N = d_in; h.K = d_out; h.lda = d_out; h.ldb = d_in; h.ldc = d_in;
  h.a_lower = true; h.alpha = 1.0f;
  return chol_gemm(L, h, w, prec);
}

LrApply lr_args(const gift_factor *f, const float *X, int d_out, int d_in, const CodecWs &w, bool inverse,
                gift_precision prec) {
  LrApply a{};
  a.terms = (prec == GIFT_PREC_TC) ? 1 : 3;
  a.X = X;
  a.U = f->U;
  a.Pc = w.Pc;
  a.sigma = f->sigma;
  a.rank = f->rank;
  a.d_out = d_out;
  a.d_in = d_in;
  a.inverse = inverse;
  a.split = (d_in % 32 == 0) ? w.split : nullptr;
  if (a.split) lr_u_planes(f->planes, w.split, d_out, d_in, &a.u_planes, &a.ut_planes);
  return a;
}

// Projection and coefficients; for shapes the tensor-core kernels take, also their operand
// planes.
cudaError_t lr_prepare(const Launch &L, const gift_factor *f, const float *X, int d_out, int d_in, const CodecWs &w,
                       bool inverse, gift_precision prec) {
  return lr_prepare_all(L, f->U, f->mu, f->sigma, f->rank, X, d_out, d_in, inverse, prec == GIFT_PREC_TC, w.part,
                        w.Pc, (d_in % 32 == 0) ? w.split : nullptr, f->planes);
}

}  // namespace

namespace gift {
void record_cuda_error(cudaError_t e) { t_last_cuda_error = e; }
}  // namespace gift

// =========================================================================================
extern "C" {

const char *gift_last_error(void) {
  return t_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(t_last_cuda_error);
}

gift_status gift_create(gift_ctx **ctx, int device) {
  if (!ctx) return GIFT_ERR_INVALID_ARG;
  *ctx = nullptr;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    return GIFT_ERR_CUDA;
  gift_ctx *c = static_cast<gift_ctx *>(std::malloc(sizeof(gift_ctx)));
  if (!c) return GIFT_ERR_CUDA;
  c->device = device;
  c->device_sms = sms;
  c->sms = sms;
  c->subspace_iters = 16;
  c->barrier_wait = kDefaultBarrierWait;
  c->sketch = 0;
  *ctx = c;
  return GIFT_OK;
}

void gift_destroy(gift_ctx *ctx) { std::free(ctx); }

gift_status gift_set_option(gift_ctx *ctx, gift_option opt, long long value) {
  if (!ctx) return GIFT_ERR_INVALID_ARG;
  if (opt == GIFT_OPT_SUBSPACE_ITERS) {
    if (value < 1 || value > 64) return GIFT_ERR_INVALID_ARG;
    ctx->subspace_iters = (int)value;
    return GIFT_OK;
  }
  if (opt == GIFT_OPT_SKETCH) {
    if (value != 0 && value != 1) return GIFT_ERR_INVALID_ARG;
    ctx->sketch = (int)value;
    return GIFT_OK;
  }
  if (opt == GIFT_OPT_BARRIER_WAIT) {
    if (value < 0 || value > 20000000000LL) return GIFT_ERR_INVALID_ARG;
    ctx->barrier_wait = value;
    return GIFT_OK;
  }
  if (opt == GIFT_OPT_SMS) {
    if (value < 1 || value > ctx->device_sms) return GIFT_ERR_INVALID_ARG;
    ctx->sms = (int)value;
    return GIFT_OK;
  }
  return GIFT_ERR_INVALID_ARG;
}

const char *gift_status_string(gift_status s) {
  switch (s) {
    case GIFT_OK: return "ok";
    case GIFT_ERR_INVALID_ARG: return "invalid argument";
    case GIFT_ERR_UNSUPPORTED: return "unsupported combination";
    case GIFT_ERR_CUDA: return "CUDA error";
    case GIFT_ERR_NONFINITE: return "non-finite value in the tensor";
    case GIFT_ERR_NOT_PD: return "factor is not positive definite";
    case GIFT_ERR_TIMEOUT: return "bounded device wait timed out";
    case GIFT_ERR_NOT_CONVERGED: return "eigensolver did not converge";
  }
  return "unknown status";
}

int gift_version(void) { return GIFT_VERSION_MAJOR * 1000 + GIFT_VERSION_MINOR; }

size_t gift_workspace_bytes(const gift_ctx *ctx, gift_op op, gift_xform kind, gift_format fmt,
                            gift_scaling scaling, int d_out, int d_in, int T, int rank) {
  (void)rank;
  if (!ctx || d_out <= 0 || d_in <= 0 || !valid_kind(kind) || !valid_fmt(fmt) || !valid_scaling(scaling))
    return (size_t)-1;
  if (op == GIFT_OP_KFAC_FACTOR)
    return T > 0 ? std::max(syrk_tc_scratch_bytes(d_in, T), syrk_planes_bytes(d_in, T)) : (size_t)-1;
  if (op == GIFT_OP_FACTOR_UPDATE) {
    if (kind == GIFT_XF_IDENTITY) return 0;
    return factor_layout(nullptr, ctx->sms, kind, d_out, d_in, T, ctx->sketch == 0).bytes;
  }
  if (op != GIFT_OP_ENCODE && op != GIFT_OP_DECODE && op != GIFT_OP_AMAX && op != GIFT_OP_REDUCE_DECODE)
    return (size_t)-1;
  return codec_layout(nullptr, ctx->sms, op, kind, d_out, d_in).bytes;
}

gift_status gift_code_sizes(gift_format fmt, gift_scaling scaling, int d_out, int d_in, size_t *code_bytes,
                            size_t *scale_count) {
  if (!code_bytes || !scale_count || d_out <= 0 || d_in <= 0 || !valid_fmt(fmt) || !valid_scaling(scaling))
    return GIFT_ERR_INVALID_ARG;
  const size_t n = (size_t)d_out * d_in;
  switch (fmt) {
    case GIFT_FMT_F32:
      *code_bytes = 4 * n;
      *scale_count = 0;
      break;
    case GIFT_FMT_NVFP4:
      if (d_in % kNvGroup) return GIFT_ERR_INVALID_ARG;
      *code_bytes = n / 2;
      *scale_count = n / kNvGroup;
      break;
    default:
      *code_bytes = n;
      *scale_count = (scaling == GIFT_SCALE_TENSOR)     ? 1
                     : (scaling == GIFT_SCALE_BLOCK512) ? (n + kBlock1d - 1) / kBlock1d
                                                        : (size_t)((d_out + kBlock - 1) / kBlock) * ((d_in + kBlock - 1) / kBlock);
  }
  return GIFT_OK;
}

// -----------------------------------------------------------------------------------------
namespace {

// A = x^T x / T (full symmetric, FP32).
//  TC precision, BF16 x: k_syrk_tc (exact products, the tensor core's accumulation over T).
//  FP32 precision with a workspace of syrk_planes_bytes: the tensor-core GEMM on the exact BF16
//    terms of x (one term for BF16 x, three for FP32 x and the six products i + j <= 2), a fresh
//    accumulator per 64 tokens summed round to nearest: FP32 accuracy.
//  Otherwise FP32 SIMT.
cudaError_t kfac_syrk(const Launch &L, const void *x, bool bf16, int T, int d, gift_precision prec, void *ws,
                      size_t ws_bytes, float *out) {
  if (prec == GIFT_PREC_TC && bf16 && ws && ws_bytes >= syrk_tc_scratch_bytes(d, T) &&
      syrk_tc_ok(d, T, x, ws, out)) {
    cudaError_t e = launch_syrk_tc(L, x, T, d, 1.0f / (float)T, ws, out);
    if (e != cudaSuccess) return e;
    return launch_mirror_lower(L, out, d);
  }
  const bool tc_planes = ws && ws_bytes >= syrk_planes_bytes(d, T) && aligned16(ws) && aligned16(out);
  if (tc_planes) {
    uint16_t *pl = static_cast<uint16_t *>(ws);
    const int rows = (d + 127) / 128 * 128, ldk = (T + 63) / 64 * 64;
    cudaError_t e;
    int nt = 3;
    (void)rows;
    (void)ldk;
    if (bf16) {   // a BF16 value is its own single term
      nt = 1;
      if ((e = launch_split_planes_bf16(L, x, d, T, d, true, pl)) != cudaSuccess) return e;
    } else if ((e = launch_split_planes(L, static_cast<const float *>(x), d, T, d, true, 3, pl)) != cudaSuccess) {
      return e;
    }
    GemmPlanes g;
    g.pa = pl;
    g.pb = pl;
    g.M = d;
    g.N = d;
    g.K = T;
    g.nta = g.ntb = nt;
    g.fp32 = true;
    g.lower_tiles = true;
    g.alpha = 1.0f / (float)T;
    g.C = out;
    g.ldc = d;
    if ((e = launch_gemm_planes(L, g)) != cudaSuccess) return e;
    return launch_mirror_lower(L, out, d);
  }
  GemmArgs g{};
  g.A = x; g.B = x; g.C = out;
  g.M = d; g.N = d; g.K = T; g.lda = d; g.ldb = d; g.ldc = d;
  g.transA = true; g.transB = false; g.a_bf16 = bf16; g.b_bf16 = bf16;
  g.lower_tiles = true; g.alpha = 1.0f / (float)T;
  cudaError_t e = launch_sgemm(L, g);
  if (e != cudaSuccess) return e;
  return launch_mirror_lower(L, out, d);
}

}  // namespace

size_t gift_factor_planes_bytes(int d_in) { return d_in > 0 ? lr_factor_planes_bytes(d_in) : (size_t)-1; }

gift_status gift_factor_prepare(gift_ctx *ctx, const gift_factor *f, cudaStream_t stream) {
  if (!ctx || !f || f->kind != GIFT_XF_LOWRANK || !f->U || !f->planes) return GIFT_ERR_INVALID_ARG;
  if (f->d_in <= 0 || f->rank < 1 || f->rank > kMaxRank || f->rank > f->d_in || !aligned16(f->planes))
    return GIFT_ERR_INVALID_ARG;
  const Launch L = mk(ctx, nullptr, stream);
  CK(launch_lr_factor_planes(L, f->U, f->d_in, f->rank, f->planes));
  return GIFT_OK;
}

gift_status gift_kfac_factor(gift_ctx *ctx, const void *a, gift_dtype a_dt, int T, int d, gift_precision prec,
                             float *A_out, void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream) {
  if (!ctx || !a || !A_out || T < 1 || d < 1) return GIFT_ERR_INVALID_ARG;
  if (a_dt != GIFT_DT_F32 && a_dt != GIFT_DT_BF16) return GIFT_ERR_INVALID_ARG;
  if (prec != GIFT_PREC_FP32 && prec != GIFT_PREC_TC) return GIFT_ERR_INVALID_ARG;
  if (prec == GIFT_PREC_TC && (!ws || ws_bytes < syrk_tc_scratch_bytes(d, T))) return GIFT_ERR_INVALID_ARG;
  const Launch L = mk(ctx, d_status, stream);
  CK(kfac_syrk(L, a, a_dt == GIFT_DT_BF16, T, d, prec, ws, ws ? ws_bytes : 0, A_out));
  return GIFT_OK;
}

// The factor refresh from activations (a, T > 0; delta for the two-sided kind) or from given
// K-FAC factors (A_in, and G_in for the two-sided kind; T = 0).
static gift_status factor_update_impl(gift_ctx *ctx, gift_factor *f, const void *a, gift_dtype a_dt, int T,
                                      const void *delta, gift_dtype d_dt, const float *A_in, const float *G_in,
                                      uint64_t seed, gift_precision prec, void *ws, size_t ws_bytes, int *d_status,
                                      cudaStream_t stream) {
  if (!ctx || !f) return GIFT_ERR_INVALID_ARG;
  if (A_in ? (a || T != 0) : (!a || T < 1)) return GIFT_ERR_INVALID_ARG;
  if (prec != GIFT_PREC_FP32 && prec != GIFT_PREC_TC) return GIFT_ERR_INVALID_ARG;
  const int d_in = f->d_in, d_out = f->d_out;
  if (d_in <= 0 || d_out <= 0) return GIFT_ERR_INVALID_ARG;
  if (!A_in && a_dt != GIFT_DT_F32 && a_dt != GIFT_DT_BF16) return GIFT_ERR_INVALID_ARG;
  if (f->kind == GIFT_XF_IDENTITY || !valid_kind(f->kind)) return GIFT_ERR_INVALID_ARG;
  gift_status cs = check_factor(f, d_out, d_in);
  if (cs != GIFT_OK) return cs;
  if (f->kind == GIFT_XF_CHOL_TWO_SIDED && !A_in && (!delta || (d_dt != GIFT_DT_F32 && d_dt != GIFT_DT_BF16)))
    return GIFT_ERR_INVALID_ARG;
  if (f->kind == GIFT_XF_CHOL_TWO_SIDED && A_in && !G_in) return GIFT_ERR_INVALID_ARG;
  const FactorWs need = factor_layout(nullptr, ctx->sms, f->kind, d_out, d_in, T, ctx->sketch == 0);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  const FactorWs w = factor_layout(ws, ctx->sms, f->kind, d_out, d_in, T, ctx->sketch == 0);
  const Launch L = mk(ctx, d_status, stream);

  // A = a^T a / T (lower tiles, then mirrored)
  auto syrk = [&](const void *x, bool bf16, int d, float *out) -> cudaError_t {
    return kfac_syrk(L, x, bf16, T, d, prec, w.at, w.at_bytes, out);
  };
  // the input-side factor: formed from the activations, or the caller's
  const float *A = A_in ? A_in : w.A;
  if (!A_in && !(f->kind == GIFT_XF_LOWRANK && w.qpl)) CK(syrk(a, a_dt == GIFT_DT_BF16, d_in, w.A));

  if (f->kind == GIFT_XF_LOWRANK && w.qpl) {
    // FP32 subspace iteration with Rayleigh-Ritz steps, the products on the tensor cores
    const int k = 64, r = f->rank;
    const bool bf16 = (a_dt == GIFT_DT_BF16);
    const int nt = (prec == GIFT_PREC_TC) ? 2 : 3;   // terms of the FP32 operands
    const bool fp32 = (prec != GIFT_PREC_TC);
    const int *skip = w.flag;
    // the activations as the A operand of Z = a Q (M = T, K = d_in): one term for BF16, split
    // into terms for FP32
    if (a) {
      if (bf16) CK(launch_split_planes_bf16(L, a, T, d_in, d_in, false, w.xpl));
      else CK(launch_split_planes(L, static_cast<const float *>(a), T, d_in, d_in, false, nt, w.xpl));
    }
    const int a_nt = bf16 ? 1 : nt;
    if (w.implicit) {
      // a^T as the A operand of Y = a^T Z / T (M = d_in, K = T), in the K-FAC workspace
      if (bf16) CK(launch_split_planes_bf16(L, a, d_in, T, d_in, true, static_cast<uint16_t *>(w.at)));
      else CK(launch_split_planes(L, static_cast<const float *>(a), d_in, T, d_in, true, nt,
                                  static_cast<uint16_t *>(w.at)));
      if (aligned16(a)) CK(launch_trace_acts32(L, a, bf16, T, d_in, w.sq, trace_partials(ctx->sms), w.tr));
      else CK(launch_trace_from_activations(L, a, bf16, T, d_in, w.sq, w.tr));
    } else {
      if (!A_in) CK(syrk(a, bf16, d_in, w.A));
      CK(launch_trace_diag(L, A, d_in, w.tr));
      CK(launch_split_planes(L, A, d_in, d_in, d_in, false, nt, w.apl));
    }
    CK(cudaMemsetAsync(w.flag, 0, sizeof(int), stream));
    auto orth = [&](float *Y, const int *sk) -> cudaError_t {   // Q = Y L^-T with Y^T Y = L L^T, twice (CholQR2)
      cudaError_t e = cudaSuccess;
      const float *src = Y;
      for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
        if ((e = launch_gram_tall(L, src, src, d_in, k, w.gparts, w.G32, true, sk)) != cudaSuccess) break;
        if ((e = launch_chol32(L, w.G32, k, w.R32, sk)) != cudaSuccess) break;
        e = launch_right_trsm64(L, src, d_in, w.R32, w.Q, sk);
        src = w.Q;
      }
      return e;
    };
    auto gemm = [&](const uint16_t *pa, int nta, const uint16_t *pb, int M, int K, float alpha, float *C, int ksplit,
                    const int *sk) -> cudaError_t {
      GemmPlanes g;
      g.pa = pa;
      g.pb = pb;
      g.M = M;
      g.N = k;
      g.K = K;
      g.nta = nta;
      g.ntb = nt;
      g.fp32 = fp32;
      g.ksplit = ksplit;
      g.parts = w.parts;
      g.alpha = alpha;
      g.C = C;
      g.ldc = k;
      g.skip = sk;
      return launch_gemm_planes(L, g);
    };
    auto za = [&](const int *sk) -> cudaError_t {   // Z = a Q
      cudaError_t e = launch_split_planes(L, w.Q, k, d_in, k, true, nt, w.qpl, sk);
      if (e != cudaSuccess) return e;
      return gemm(w.xpl, a_nt, w.qpl, T, d_in, 1.0f, w.Z, 1, sk);
    };
    auto sketch = [&](const int *sk) -> cudaError_t {   // Y = A Q
      cudaError_t e;
      if (w.implicit) {   // A Q = a^T (a Q) / T
        if ((e = za(sk)) != cudaSuccess) return e;
        if ((e = launch_split_planes(L, w.Z, k, T, k, true, nt, w.zpl, sk)) != cudaSuccess) return e;
        e = gemm(static_cast<const uint16_t *>(w.at), a_nt, w.zpl, d_in, T, 1.0f / (float)T, w.Y, w.ksplit, sk);
      } else {
        if ((e = launch_split_planes(L, w.Q, k, d_in, k, true, nt, w.qpl, sk)) != cudaSuccess) return e;
        e = gemm(w.apl, nt, w.qpl, d_in, d_in, 1.0f, w.Y, w.ksplit, sk);
      }
      return e;
    };
    auto ritz = [&](const int *sk) -> cudaError_t {   // B = Q^T Y; (theta, V) = eig(B); Y <- Y V
      cudaError_t e = launch_gram_tall(L, w.Q, w.Y, d_in, k, w.gparts, w.B32, true, sk);
      if (e != cudaSuccess) return e;
      // the Ritz directions condition the next CholQR: a few sweeps are enough
      if ((e = launch_jacobi32(L, w.B32, k, w.th, w.V32, 2, false, sk)) != cudaSuccess) return e;
      if ((e = launch_ritz_rotate(L, w.Y, w.Q, d_in, w.V32, w.th, w.rparts, sk)) != cudaSuccess) return e;
      return launch_ritz_check(L, w.rparts, ritz_rotate_ctas(ctx->sms, d_in), w.th, r, w.flag);
    };
    CK(launch_philox_gaussian(L, w.Y, (size_t)d_in * k, seed));
    CK(orth(w.Y, nullptr));
    for (int it = 0; it < ctx->subspace_iters; ++it) {
      CK(sketch(skip));
      // Rayleigh-Ritz on the first two iterations (the random start gives a badly conditioned
      // A Q), then every fourth with the convergence test; in between the basis stays close to
      // the Ritz directions, so A Q keeps nearly orthogonal columns
      if (it < 2 || it % 4 == 3) CK(ritz(skip));
      CK(orth(w.Y, skip));
    }
    // final Rayleigh-Ritz step from the activations: B = Q^T A Q = (a Q)^T (a Q) / T, a Gram
    // matrix (no cancellation between large and small eigenvalues), solved to convergence;
    // from a given A, B = Q^T (A Q)
    if (a) {
      CK(za(nullptr));
      CK(launch_gram_tall(L, w.Z, w.Z, T, k, w.gparts, w.B32, true, nullptr, 1.0f / (float)T));
    } else {
      CK(sketch(nullptr));
      CK(launch_gram_tall(L, w.Q, w.Y, d_in, k, w.gparts, w.B32, true, nullptr));
    }
    CK(launch_jacobi32(L, w.B32, k, w.th, w.V32, 40, true, nullptr));
    CK(launch_f32_to_f64(L, w.V32, w.V, (size_t)k * k));
    CK(launch_f32_to_f64(L, w.th, w.ev, (size_t)k));
    CK(launch_lowrank_outputs(L, w.Q, d_in, k, w.V, w.ev, w.tr, r, f->U, f->mu, f->sigma));
    if (f->planes) CK(launch_lr_factor_planes(L, f->U, d_in, r, f->planes));
    return GIFT_OK;
  }

  if (f->kind == GIFT_XF_LOWRANK) {
    const int k = w.k;
    if (a) CK(launch_trace_from_activations(L, a, a_dt == GIFT_DT_BF16, T, d_in, w.sq, w.tr));
    else CK(launch_trace_diag(L, A, d_in, w.tr));
    auto cholqr = [&](const float *in, float *out) -> cudaError_t {
      DgemmArgs g{};
      g.A = in; g.B = in; g.C = w.Gp;
      g.M = k; g.N = k; g.K = d_in; g.lda = k; g.ldb = k; g.ldc = k;
      g.transA = true; g.transB = false; g.a_f32 = true; g.b_f32 = true;
      g.alpha = 1.0; g.beta = 0.0; g.splits = w.gsplits; g.slice_stride = (size_t)k * k;
      cudaError_t e = launch_dgemm(L, g);
      if (e != cudaSuccess) return e;
      if ((e = launch_sum_slices(L, w.Gp, w.gsplits, (size_t)k * k, (size_t)k * k, w.G, 1.0)) != cudaSuccess) return e;
      if ((e = launch_small_chol_rinv(L, w.G, k, w.Rinv)) != cudaSuccess) return e;
      DgemmArgs q{};
      q.A = in; q.B = w.Rinv; q.C = w.Q64;
      q.M = d_in; q.N = k; q.K = k; q.lda = k; q.ldb = k; q.ldc = k;
      q.a_f32 = true; q.b_f32 = false; q.alpha = 1.0; q.beta = 0.0; q.splits = 1;
      if ((e = launch_dgemm(L, q)) != cudaSuccess) return e;
      return launch_f64_to_f32(L, w.Q64, out, (size_t)d_in * k, false, k);
    };
    auto aq = [&]() -> cudaError_t {   // Y = A Q
      GemmArgs g{};
      g.A = A; g.B = w.Q; g.C = w.Y;
      g.M = d_in; g.N = k; g.K = d_in; g.lda = d_in; g.ldb = k; g.ldc = k; g.alpha = 1.0f;
      return launch_sgemm_splitk(L, g, w.yparts, w.ysplits);
    };
    if (k == d_in) {
      CK(launch_eye(L, w.Q, k));
      CK(launch_f32_to_f64(L, A, w.G, (size_t)k * k));
    } else {
      CK(launch_philox_gaussian(L, w.Y, (size_t)d_in * k, seed));
      CK(cholqr(w.Y, w.Q));
      CK(cholqr(w.Q, w.Q));
      for (int it = 0; it < ctx->subspace_iters; ++it) {
        CK(aq());
        CK(cholqr(w.Y, w.Q));
        CK(cholqr(w.Q, w.Q));
      }
      CK(aq());
      DgemmArgs g{};   // B = Q^T (A Q)
      g.A = w.Q; g.B = w.Y; g.C = w.Gp;
      g.M = k; g.N = k; g.K = d_in; g.lda = k; g.ldb = k; g.ldc = k;
      g.transA = true; g.a_f32 = true; g.b_f32 = true;
      g.alpha = 1.0; g.beta = 0.0; g.splits = w.gsplits; g.slice_stride = (size_t)k * k;
      CK(launch_dgemm(L, g));
      CK(launch_sum_slices(L, w.Gp, w.gsplits, (size_t)k * k, (size_t)k * k, w.G, 1.0));
    }
    CK(launch_jacobi(L, w.G, k, w.ev, w.V));
    CK(launch_lowrank_outputs(L, w.Q, d_in, k, w.V, w.ev, w.tr, f->rank, f->U, f->mu, f->sigma));
    if (f->planes) CK(launch_lr_factor_planes(L, f->U, d_in, f->rank, f->planes));
    return GIFT_OK;
  }

  // Cholesky variants
  const size_t nn = (size_t)d_in * d_in;
  CK(launch_f32_to_f64(L, A, w.A64, nn));
  CK(launch_chol_inv(L, w.A64, w.Ai64, d_in, w.work));
  CK(launch_f64_to_f32(L, w.A64, f->LA, nn, true, d_in));
  CK(launch_f64_to_f32(L, w.Ai64, f->LAinv, nn, true, d_in));
  if (f->kind == GIFT_XF_CHOL_TWO_SIDED) {
    const size_t mm = (size_t)d_out * d_out;
    if (!G_in) CK(syrk(delta, d_dt == GIFT_DT_BF16, d_out, w.Gf));
    CK(launch_f32_to_f64(L, G_in ? G_in : w.Gf, w.G64, mm));
    CK(launch_chol_inv(L, w.G64, w.Gi64, d_out, w.work));
    CK(launch_f64_to_f32(L, w.G64, f->LG, mm, true, d_out));
    CK(launch_f64_to_f32(L, w.Gi64, f->LGinv, mm, true, d_out));
  }
  return GIFT_OK;
}

gift_status gift_factor_update(gift_ctx *ctx, gift_factor *f, const void *a, gift_dtype a_dt, int T,
                               const void *delta, gift_dtype d_dt, uint64_t seed, gift_precision prec,
                               void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream) {
  if (!a || T < 1) return GIFT_ERR_INVALID_ARG;
  return factor_update_impl(ctx, f, a, a_dt, T, delta, d_dt, nullptr, nullptr, seed, prec, ws, ws_bytes, d_status,
                            stream);
}

gift_status gift_factor_update_from_kfac(gift_ctx *ctx, gift_factor *f, const float *A, const float *G,
                                         uint64_t seed, gift_precision prec, void *ws, size_t ws_bytes,
                                         int *d_status, cudaStream_t stream) {
  if (!A) return GIFT_ERR_INVALID_ARG;
  return factor_update_impl(ctx, f, nullptr, GIFT_DT_F32, 0, nullptr, GIFT_DT_F32, A, G, seed, prec, ws, ws_bytes,
                            d_status, stream);
}

// -----------------------------------------------------------------------------------------
static gift_status codec_common_checks(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in,
                                       gift_format fmt, gift_scaling scaling) {
  if (!ctx || !W || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if (!valid_fmt(fmt) || !valid_scaling(scaling)) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && d_in % kNvGroup) return GIFT_ERR_INVALID_ARG;
  const gift_status fs = check_factor(f, d_out, d_in);
  if (fs != GIFT_OK) return fs;
  if (scaling == GIFT_SCALE_BLOCK512 && fmt != GIFT_FMT_NVFP4 && fmt != GIFT_FMT_F32 && kind_of(f) == GIFT_XF_LOWRANK)
    return GIFT_ERR_UNSUPPORTED;
  return GIFT_OK;
}

static gift_status encode_checks(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in,
                                 gift_format fmt, gift_scaling scaling, const float *residual, const void *codes,
                                 const void *scales, const float *tensor_scale, const void *ws, size_t ws_bytes) {
  gift_status cs = codec_common_checks(ctx, f, W, d_out, d_in, fmt, scaling);
  if (cs != GIFT_OK) return cs;
  if (!codes) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_F32 && !scales) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && !tensor_scale) return GIFT_ERR_INVALID_ARG;
  if (residual == W || codes == (const void *)W) return GIFT_ERR_INVALID_ARG;
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_ENCODE, kind_of(f), d_out, d_in);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  return GIFT_OK;
}

// The batched rank-r encode of nb tensors sharing f (per-tensor FP8 or NVFP4, no residual):
// false when the shape or a pointer does not qualify, with nothing enqueued.
// amax_only: the same transform, its amax max-accumulated into each item's amax_out (the
// amax gift_encode would use, for the shapes gift_encode sends here).
static bool try_batch(gift_ctx *ctx, const gift_factor *f, int d_out, int d_in, gift_format fmt,
                        gift_precision prec, const CodecWs &w, const Launch &L, int nb, const LrEncodeItem *items,
                        gift_status *st, bool amax_only = false) {
  if (!w.bpart || !w.bplanes) return false;
  LrApply o = lr_args(f, items[0].X, d_out, d_in, w, false, prec);
  o.amax_ws = w.amax;   // one word per tensor, then the grid-barrier counter
  o.grid_counter = reinterpret_cast<unsigned int *>(w.amax + kEncodeBatchMax);
  const int epi = (fmt == GIFT_FMT_NVFP4) ? LR_NVFP4 : LR_PACK_TENSOR;
  for (int k = 0; k < nb; ++k) {
    LrApply ok = o;
    ok.X = items[k].X;
    if (!lr_encode_batch_ok(L, ok, epi)) return false;
  }
  *st = GIFT_OK;
  cudaError_t e = cudaSuccess;
  if (!f->planes) e = launch_lr_split_u_all(L, f->U, d_out, d_in, f->rank, prec == GIFT_PREC_TC ? 1 : 2, w.split);
  for (int k0 = 0; k0 < nb && e == cudaSuccess; k0 += kBatchWs) {
    const int m = (nb - k0 < kBatchWs) ? nb - k0 : kBatchWs;
    e = cudaMemsetAsync(w.amax, 0, (kEncodeBatchMax + 1) * sizeof(float), L.stream);   // amax words + counter
    if (e == cudaSuccess)
      e = launch_lr_encode_batch(L, amax_only ? LR_AMAX : epi, fmt, o, f->mu, w.bpart, w.bplanes, m, items + k0);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    *st = GIFT_ERR_CUDA;
  }
  return true;
}

gift_status gift_amax(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in, gift_format fmt,
                      gift_scaling scaling, gift_precision prec, const float *residual, float *amax_accum, void *ws,
                      size_t ws_bytes, int *d_status, cudaStream_t stream) {
  gift_status cs = codec_common_checks(ctx, f, W, d_out, d_in, fmt, scaling);
  if (cs != GIFT_OK) return cs;
  if (!amax_accum || fmt == GIFT_FMT_F32) return GIFT_ERR_INVALID_ARG;
  const gift_xform kind = kind_of(f);
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_AMAX, kind, d_out, d_in);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_AMAX, kind, d_out, d_in);
  const Launch L = mk(ctx, d_status, stream);
  const bool block = (fmt != GIFT_FMT_NVFP4 && scaling == GIFT_SCALE_BLOCK128);
  const bool b512 = (fmt != GIFT_FMT_NVFP4 && scaling == GIFT_SCALE_BLOCK512);
  const size_t n = (size_t)d_out * d_in;
  if (kind == GIFT_XF_LOWRANK) {
    if (!block && !residual) {
      // the kernel (and so the arithmetic) gift_encode uses for this shape
      LrEncodeItem it;
      std::memset(&it, 0, sizeof(it));
      it.X = W;
      it.amax_out = amax_accum;
      gift_status st = GIFT_OK;
      if (try_batch(ctx, f, d_out, d_in, fmt, prec, w, L, 1, &it, &st, true)) return st;
    }
    CK(lr_prepare(L, f, W, d_out, d_in, w, false, prec));
    LrApply a = lr_args(f, W, d_out, d_in, w, false, prec);
    a.R = const_cast<float *>(residual);   // read only by the amax epilogue
    a.amax_ws = amax_accum;
    CK(launch_lr_apply(L, block ? LR_BLOCK_AMAX : LR_AMAX, fmt, a));
    return GIFT_OK;
  }
  const float *src = W;
  if (kind != GIFT_XF_IDENTITY) {
    CK(chol_whiten(L, f, W, d_out, d_in, w, prec));
    src = w.xbuf;
  }
  if (block) CK(launch_block128(L, fmt, 1, src, const_cast<float *>(residual), d_out, d_in, nullptr, nullptr,
                                nullptr, amax_accum, nullptr, nullptr));
  else if (b512) CK(launch_block512(L, fmt, 1, src, const_cast<float *>(residual), n, nullptr, nullptr, nullptr,
                                    amax_accum, nullptr, nullptr));
  else CK(launch_amax(L, src, residual, n, amax_accum));
  return GIFT_OK;
}

gift_status gift_encode(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out, int d_in, gift_format fmt,
                        gift_scaling scaling, gift_precision prec, const float *amax_in, float *residual,
                        void *codes, void *scales, float *tensor_scale, float *transformed_out, float *amax_out,
                        void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream) {
  gift_status cs = encode_checks(ctx, f, W, d_out, d_in, fmt, scaling, residual, codes, scales, tensor_scale, ws,
                                 ws_bytes);
  if (cs != GIFT_OK) return cs;
  const gift_xform kind = kind_of(f);
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_ENCODE, kind, d_out, d_in);
  const Launch L = mk(ctx, d_status, stream);
  const size_t n = (size_t)d_out * d_in;
  uint8_t *c8 = static_cast<uint8_t *>(codes);
  const bool block = (scaling == GIFT_SCALE_BLOCK128);

  if (kind == GIFT_XF_LOWRANK) {
    if (fmt != GIFT_FMT_F32 && !(fmt != GIFT_FMT_NVFP4 && block) && !residual) {
      // the batched kernels (projection pass, then apply and pack with the tensor on chip)
      // where the shape fits
      LrEncodeItem it;
      it.X = W;
      it.codes = c8;
      it.scales = scales;
      it.tscale = tensor_scale;
      it.amax_out = amax_out;
      it.tout = transformed_out;
      it.amax_in = amax_in;
      gift_status st = GIFT_OK;
      if (try_batch(ctx, f, d_out, d_in, fmt, prec, w, L, 1, &it, &st)) return st;
    }
    CK(lr_prepare(L, f, W, d_out, d_in, w, false, prec));
    LrApply a = lr_args(f, W, d_out, d_in, w, false, prec);
    a.R = residual;
    if (fmt == GIFT_FMT_F32) {
      a.out = static_cast<float *>(codes);
      CK(launch_lr_apply(L, LR_STORE, fmt, a));
      if (transformed_out) CK(cudaMemcpyAsync(transformed_out, codes, n * 4, cudaMemcpyDeviceToDevice, stream));
      if (residual) CK(cudaMemsetAsync(residual, 0, n * 4, stream));
      return GIFT_OK;
    }
    a.tout = transformed_out;
    a.codes = c8;
    a.scales = scales;
    a.tscale = tensor_scale;
    a.amax_out = amax_out;
    a.amax_in = amax_in;
    if (fmt != GIFT_FMT_NVFP4 && block) {
      CK(launch_lr_apply(L, LR_BLOCK, fmt, a));
      return GIFT_OK;
    }
    const int epi = (fmt == GIFT_FMT_NVFP4) ? LR_NVFP4 : LR_PACK_TENSOR;
    if (!amax_in) CK(cudaMemsetAsync(w.amax, 0, sizeof(float), stream));
    a.amax_ws = w.amax;
    a.grid_counter = reinterpret_cast<unsigned int *>(w.amax + 16);
    if (lr_encode_fused_ok(L, a, epi)) {
      // one pass over W: transform, grid-wide amax and pack with W~ held on chip
      CK(cudaMemsetAsync(a.grid_counter, 0, sizeof(unsigned int), stream));
      CK(launch_lr_encode_fused(L, epi, fmt, a));
      return GIFT_OK;
    }
    if (!amax_in) {
      LrApply am = a;
      am.tout = nullptr;
      CK(launch_lr_apply(L, LR_AMAX, fmt, am));
    }
    CK(launch_lr_apply(L, epi, fmt, a));
    return GIFT_OK;
  }

  const float *src = W;
  if (kind != GIFT_XF_IDENTITY) {
    CK(chol_whiten(L, f, W, d_out, d_in, w, prec));
    src = w.xbuf;
  }
  if (fmt == GIFT_FMT_F32) {
    CK(launch_pack_f32(L, src, residual, n, static_cast<float *>(codes), transformed_out));
    return GIFT_OK;
  }
  if (fmt != GIFT_FMT_NVFP4 && block) {
    CK(launch_block128(L, fmt, 0, src, residual, d_out, d_in, amax_in, c8, static_cast<float *>(scales), amax_out,
                       transformed_out, nullptr));
    return GIFT_OK;
  }
  if (fmt != GIFT_FMT_NVFP4 && scaling == GIFT_SCALE_BLOCK512) {
    CK(launch_block512(L, fmt, 0, src, residual, n, amax_in, c8, static_cast<float *>(scales), amax_out,
                       transformed_out, nullptr));
    return GIFT_OK;
  }
  const float *amax = amax_in;
  if (!amax) {
    CK(cudaMemsetAsync(w.amax, 0, sizeof(float), stream));
    CK(launch_amax(L, src, residual, n, w.amax));
    amax = w.amax;
  }
  if (fmt == GIFT_FMT_NVFP4)
    CK(launch_pack_nvfp4(L, src, residual, n, amax, c8, static_cast<uint8_t *>(scales), tensor_scale, amax_out,
                         transformed_out));
  else
    CK(launch_pack_tensor(L, fmt, src, residual, n, amax, c8, static_cast<float *>(scales), amax_out,
                          transformed_out));
  return GIFT_OK;
}

gift_status gift_encode_replicas(gift_ctx *ctx, const gift_factor *f, int R, const float *const *W, int d_out,
                                 int d_in, gift_format fmt, gift_scaling scaling, gift_precision prec,
                                 const float *const *amax_in, void *const *codes, void *const *scales,
                                 float *const *tensor_scales, float *const *amax_out, void *ws, size_t ws_bytes,
                                 int *d_status, cudaStream_t stream) {
  if (!ctx || !W || !codes || R < 1 || R > kMaxReplicas) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_F32 && !scales) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && !tensor_scales) return GIFT_ERR_INVALID_ARG;
  auto at = [](auto arr, int r) { return arr ? arr[r] : nullptr; };
  // every replica is checked before anything is enqueued
  for (int r = 0; r < R; ++r) {
    const gift_status cs = encode_checks(ctx, f, W[r], d_out, d_in, fmt, scaling, nullptr, codes[r], at(scales, r),
                                         at(tensor_scales, r), ws, ws_bytes);
    if (cs != GIFT_OK) return cs;
  }
  const gift_xform kind = kind_of(f);
  const Launch L = mk(ctx, d_status, stream);
  if (kind == GIFT_XF_LOWRANK && fmt != GIFT_FMT_F32 && !(fmt != GIFT_FMT_NVFP4 && scaling != GIFT_SCALE_TENSOR)) {
    const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_ENCODE, kind, d_out, d_in);
    LrEncodeItem items[kMaxReplicas];
    for (int r = 0; r < R; ++r) {
      items[r].X = W[r];
      items[r].codes = static_cast<uint8_t *>(codes[r]);
      items[r].scales = at(scales, r);
      items[r].tscale = at(tensor_scales, r);
      items[r].amax_out = at(amax_out, r);
      items[r].tout = nullptr;
      items[r].amax_in = at(amax_in, r);
    }
    gift_status st = GIFT_OK;
    if (try_batch(ctx, f, d_out, d_in, fmt, prec, w, L, R, items, &st)) return st;
  }
  if (kind == GIFT_XF_IDENTITY && (fmt == GIFT_FMT_E4M3 || fmt == GIFT_FMT_E5M2) && scaling == GIFT_SCALE_TENSOR) {
    // one streaming launch for the replicas' own amax (those without a caller amax), one for
    // the pack
    const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_ENCODE, kind, d_out, d_in);
    const size_t n = (size_t)d_out * d_in;
    MultiArgs m;
    std::memset(&m, 0, sizeof(m));
    MultiArgs own;
    std::memset(&own, 0, sizeof(own));
    int nown = 0;
    for (int r = 0; r < R; ++r) {
      m.x[r] = W[r];
      m.codes[r] = static_cast<uint8_t *>(codes[r]);
      m.scale[r] = static_cast<float *>(scales[r]);
      m.amax_out[r] = at(amax_out, r);
      m.amax_in[r] = at(amax_in, r);
      if (!m.amax_in[r]) {
        m.amax_in[r] = w.amax + r;   // the workspace holds 64 amax words
        own.x[nown] = W[r];
        own.amax_bits[nown++] = reinterpret_cast<uint32_t *>(w.amax + r);
      }
    }
    if (multi_ok(m, R, n, true)) {
      if (nown) {
        CK(cudaMemsetAsync(w.amax, 0, (size_t)R * sizeof(float), stream));
        CK(launch_amax_multi(L, own, nown, n));
      }
      CK(launch_pack_tensor_multi(L, fmt, m, R, n));
      return GIFT_OK;
    }
  }
  for (int r = 0; r < R; ++r) {
    const gift_status st = gift_encode(ctx, f, W[r], d_out, d_in, fmt, scaling, prec, at(amax_in, r), nullptr,
                                       codes[r], at(scales, r), at(tensor_scales, r), nullptr, at(amax_out, r), ws,
                                       ws_bytes, d_status, stream);
    if (st != GIFT_OK) return st;
  }
  return GIFT_OK;
}

// Workspace control words 62 and 63: the shared amax and the barrier count of the
// shared-scale encode.  Nothing else in that call touches them: the batched rank-r encode
// uses words 0-16, and the replicas are encoded with the shared word as their amax, so no
// replica's own-amax word is used.
constexpr int kSharedAmaxWord = 62;

gift_status gift_encode_replicas_shared(gift_ctx *ctx, const gift_factor *f, int R, const float *const *W,
                                        int d_out, int d_in, gift_format fmt, gift_scaling scaling,
                                        gift_precision prec, void *const *codes, void *const *scales,
                                        float *const *tensor_scales, float *shared_amax_out, void *ws,
                                        size_t ws_bytes, int *d_status, cudaStream_t stream) {
  if (!ctx || !W || !codes || !scales || R < 1 || R > kMaxReplicas) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_F32) return GIFT_ERR_INVALID_ARG;   // no scale to share
  if (fmt != GIFT_FMT_NVFP4 && scaling != GIFT_SCALE_TENSOR) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && !tensor_scales) return GIFT_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r) {
    const gift_status cs = encode_checks(ctx, f, W[r], d_out, d_in, fmt, scaling, nullptr, codes[r], scales[r],
                                         tensor_scales ? tensor_scales[r] : nullptr, ws, ws_bytes);
    if (cs != GIFT_OK) return cs;
  }
  const gift_xform kind = kind_of(f);
  const Launch L = mk(ctx, d_status, stream);
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_ENCODE, kind, d_out, d_in);
  float *word = w.amax + kSharedAmaxWord;
  const size_t n = (size_t)d_out * d_in;
  if (kind == GIFT_XF_IDENTITY && fmt != GIFT_FMT_NVFP4) {
    MultiArgs m;
    std::memset(&m, 0, sizeof(m));
    for (int r = 0; r < R; ++r) {
      m.x[r] = W[r];
      m.codes[r] = static_cast<uint8_t *>(codes[r]);
      m.scale[r] = static_cast<float *>(scales[r]);
    }
    if (multi_ok(m, R, n, true)) {
      CK(cudaMemsetAsync(word, 0, 2 * sizeof(float), stream));   // amax bits, barrier count
      CK(launch_encode_shared(L, fmt, m, R, n, reinterpret_cast<uint32_t *>(word), shared_amax_out));
      return GIFT_OK;
    }
  }
  // any other kind, format or layout: the shared amax, then every replica encoded with it
  CK(cudaMemsetAsync(word, 0, sizeof(float), stream));
  gift_status st = gift_amax_replicas(ctx, f, R, W, d_out, d_in, fmt, scaling, prec, word, ws, ws_bytes, d_status,
                                      stream);
  if (st != GIFT_OK) return st;
  const float *ain[kMaxReplicas];
  for (int r = 0; r < R; ++r) ain[r] = word;
  st = gift_encode_replicas(ctx, f, R, W, d_out, d_in, fmt, scaling, prec, ain, codes, scales, tensor_scales,
                            nullptr, ws, ws_bytes, d_status, stream);
  if (st != GIFT_OK) return st;
  if (shared_amax_out) CK(cudaMemcpyAsync(shared_amax_out, word, sizeof(float), cudaMemcpyDeviceToDevice, stream));
  return GIFT_OK;
}

gift_status gift_amax_replicas(gift_ctx *ctx, const gift_factor *f, int R, const float *const *W, int d_out,
                               int d_in, gift_format fmt, gift_scaling scaling, gift_precision prec,
                               float *amax_accum, void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream) {
  if (!ctx || !W || !amax_accum || R < 1 || R > kMaxReplicas || fmt == GIFT_FMT_F32) return GIFT_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r) {
    const gift_status cs = codec_common_checks(ctx, f, W[r], d_out, d_in, fmt, scaling);
    if (cs != GIFT_OK) return cs;
  }
  const gift_xform kind = kind_of(f);
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_AMAX, kind, d_out, d_in);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  const Launch L = mk(ctx, d_status, stream);
  const bool block = (fmt != GIFT_FMT_NVFP4 && scaling != GIFT_SCALE_TENSOR);
  if (!block && kind == GIFT_XF_IDENTITY) {
    MultiArgs m;
    std::memset(&m, 0, sizeof(m));
    for (int r = 0; r < R; ++r) {
      m.x[r] = W[r];
      m.amax_bits[r] = reinterpret_cast<uint32_t *>(amax_accum);
    }
    if (multi_ok(m, R, (size_t)d_out * d_in, false)) {
      CK(launch_amax_multi(L, m, R, (size_t)d_out * d_in));
      return GIFT_OK;
    }
  }
  if (!block && kind == GIFT_XF_LOWRANK) {
    const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_AMAX, kind, d_out, d_in);
    LrEncodeItem items[kMaxReplicas];
    std::memset(items, 0, sizeof(items));
    for (int r = 0; r < R; ++r) {
      items[r].X = W[r];
      items[r].amax_out = amax_accum;   // max-accumulated by every replica
    }
    gift_status st = GIFT_OK;
    if (try_batch(ctx, f, d_out, d_in, fmt, prec, w, L, R, items, &st, true)) return st;
  }
  for (int r = 0; r < R; ++r) {
    const gift_status st = gift_amax(ctx, f, W[r], d_out, d_in, fmt, scaling, prec, nullptr, amax_accum, ws,
                                     ws_bytes, d_status, stream);
    if (st != GIFT_OK) return st;
  }
  return GIFT_OK;
}

gift_status gift_replica_reduce(gift_ctx *ctx, int R, const void *const *codes, const void *const *scales,
                                const float *const *tensor_scales, gift_format fmt, gift_scaling scaling, int d_out,
                                int d_in, float *avg_out, int *d_status, cudaStream_t stream) {
  if (!ctx || !codes || !avg_out || R < 1 || R > kMaxReplicas || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if (!valid_fmt(fmt) || !valid_scaling(scaling)) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && (d_in % kNvGroup || !tensor_scales)) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_F32 && !scales) return GIFT_ERR_INVALID_ARG;
  ReduceArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < R; ++r) {
    if (!codes[r]) return GIFT_ERR_INVALID_ARG;
    a.codes[r] = codes[r];
    if (fmt != GIFT_FMT_F32) {
      if (!scales[r]) return GIFT_ERR_INVALID_ARG;
      a.scales[r] = scales[r];
    }
    if (fmt == GIFT_FMT_NVFP4) {
      if (!tensor_scales[r]) return GIFT_ERR_INVALID_ARG;
      a.tscales[r] = tensor_scales[r];
    }
  }
  const Launch L = mk(ctx, d_status, stream);
  CK(launch_reduce(L, a, R, fmt, scaling, d_out, d_in, avg_out));
  return GIFT_OK;
}

gift_status gift_decode(gift_ctx *ctx, const gift_factor *f, const void *in, int in_is_codes, const void *scales,
                        const float *tensor_scale, gift_format fmt, gift_scaling scaling, gift_precision prec,
                        int d_out, int d_in, float *W_out, void *ws, size_t ws_bytes, int *d_status,
                        cudaStream_t stream) {
  if (!ctx || !in || !W_out || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if ((const void *)W_out == in) return GIFT_ERR_INVALID_ARG;
  const bool codes_in = in_is_codes && fmt != GIFT_FMT_F32;
  if (in_is_codes && (!valid_fmt(fmt) || !valid_scaling(scaling))) return GIFT_ERR_INVALID_ARG;
  if (codes_in && !scales) return GIFT_ERR_INVALID_ARG;
  if (codes_in && fmt == GIFT_FMT_NVFP4 && (d_in % kNvGroup || !tensor_scale)) return GIFT_ERR_INVALID_ARG;
  gift_status cs = check_factor(f, d_out, d_in);
  if (cs != GIFT_OK) return cs;
  const gift_xform kind = kind_of(f);
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_DECODE, kind, d_out, d_in);
  if (need.bytes && (!ws || ws_bytes < need.bytes)) return GIFT_ERR_INVALID_ARG;
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_DECODE, kind, d_out, d_in);
  const Launch L = mk(ctx, d_status, stream);
  const size_t n = (size_t)d_out * d_in;

  // 1. the whitened tensor X in FP32
  const float *X = static_cast<const float *>(in);
  if (codes_in) {
    float *dst = (kind == GIFT_XF_IDENTITY) ? W_out : w.xbuf;
    ReduceArgs a;
    std::memset(&a, 0, sizeof(a));
    a.codes[0] = in;
    a.scales[0] = scales;
    a.tscales[0] = tensor_scale;
    CK(launch_reduce(L, a, 1, fmt, scaling, d_out, d_in, dst));
    if (kind == GIFT_XF_IDENTITY) return GIFT_OK;
    X = w.xbuf;
  }
  // 2. map back
  if (kind == GIFT_XF_IDENTITY) {
    CK(launch_pack_f32(L, X, nullptr, n, W_out, nullptr));
  } else if (kind == GIFT_XF_LOWRANK) {
    CK(lr_prepare(L, f, X, d_out, d_in, w, true, prec));
    LrApply a = lr_args(f, X, d_out, d_in, w, true, prec);
    a.out = W_out;
    CK(launch_lr_apply(L, LR_STORE, GIFT_FMT_F32, a));
  } else {
    CK(chol_unwhiten(L, f, X, d_out, d_in, W_out, w, prec));
  }
  return GIFT_OK;
}

gift_status gift_reduce_decode(gift_ctx *ctx, const gift_factor *f, int R, const void *const *codes,
                               const void *const *scales, const float *const *tensor_scales, gift_format fmt,
                               gift_scaling scaling, gift_precision prec, int d_out, int d_in, float *avg_out,
                               float *W_out, void *ws, size_t ws_bytes, int *d_status, cudaStream_t stream) {
  if (!ctx || !codes || !W_out || R < 1 || R > kMaxReplicas || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if (!valid_fmt(fmt) || !valid_scaling(scaling)) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_F32 && !scales) return GIFT_ERR_INVALID_ARG;
  if (fmt == GIFT_FMT_NVFP4 && (d_in % kNvGroup || !tensor_scales)) return GIFT_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r)
    if (!codes[r] || (fmt != GIFT_FMT_F32 && !scales[r]) || (fmt == GIFT_FMT_NVFP4 && !tensor_scales[r]) ||
        codes[r] == (const void *)W_out || codes[r] == (const void *)avg_out)
      return GIFT_ERR_INVALID_ARG;
  if (avg_out && avg_out == W_out) return GIFT_ERR_INVALID_ARG;
  gift_status cs = check_factor(f, d_out, d_in);
  if (cs != GIFT_OK) return cs;
  const gift_xform kind = kind_of(f);
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_REDUCE_DECODE, kind, d_out, d_in);
  if (need.bytes && (!ws || ws_bytes < need.bytes)) return GIFT_ERR_INVALID_ARG;
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_REDUCE_DECODE, kind, d_out, d_in);
  // The average goes to avg_out or to the workspace's own buffer, back to back with the decode,
  // which then reads it from L2 (a 1536 x 6144 average, 38 MB, stays resident).  The decode of
  // an FP32 input uses the decode workspace's partials and planes, which this layout places
  // before its average buffer.
  float *X = avg_out ? avg_out : (kind == GIFT_XF_IDENTITY ? W_out : w.rdavg);
  gift_status st = gift_replica_reduce(ctx, R, codes, scales, tensor_scales, fmt, scaling, d_out, d_in, X, d_status,
                                       stream);
  if (st != GIFT_OK || X == W_out) return st;
  return gift_decode(ctx, f, X, 0, nullptr, nullptr, GIFT_FMT_F32, GIFT_SCALE_TENSOR, prec, d_out, d_in, W_out, ws,
                     ws_bytes, d_status, stream);
}

gift_status gift_boundary_hit_rate(gift_ctx *ctx, const float *W, int d_out, int d_in, gift_format fmt,
                                   gift_scaling scaling, unsigned long long *d_counts, void *ws, size_t ws_bytes,
                                   int *d_status, cudaStream_t stream) {
  if (!ctx || !W || !d_counts || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_E4M3 && fmt != GIFT_FMT_E5M2) return GIFT_ERR_INVALID_ARG;
  if (!valid_scaling(scaling)) return GIFT_ERR_INVALID_ARG;
  const Launch L = mk(ctx, d_status, stream);
  if (scaling == GIFT_SCALE_BLOCK128) {
    CK(launch_block128(L, fmt, 2, W, nullptr, d_out, d_in, nullptr, nullptr, nullptr, nullptr, nullptr, d_counts));
    return GIFT_OK;
  }
  if (scaling == GIFT_SCALE_BLOCK512) {
    CK(launch_block512(L, fmt, 2, W, nullptr, (size_t)d_out * d_in, nullptr, nullptr, nullptr, nullptr, nullptr,
                       d_counts));
    return GIFT_OK;
  }
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_AMAX, GIFT_XF_IDENTITY, d_out, d_in);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_AMAX, GIFT_XF_IDENTITY, d_out, d_in);
  const size_t n = (size_t)d_out * d_in;
  CK(cudaMemsetAsync(w.amax, 0, sizeof(float), stream));
  CK(launch_amax(L, W, nullptr, n, w.amax));
  CK(launch_hits_tensor(L, fmt, W, n, w.amax, d_counts));
  return GIFT_OK;
}

gift_status gift_boundary_hit_rates(gift_ctx *ctx, int n_tensors, const float *const *W, const int *d_out,
                                    const int *d_in, gift_format fmt, gift_scaling scaling,
                                    unsigned long long *d_counts, void *ws, size_t ws_bytes, int *d_status,
                                    cudaStream_t stream) {
  if (!ctx || !W || !d_out || !d_in || !d_counts || n_tensors < 1) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_E4M3 && fmt != GIFT_FMT_E5M2) return GIFT_ERR_INVALID_ARG;
  if (!valid_scaling(scaling)) return GIFT_ERR_INVALID_ARG;
  for (int t = 0; t < n_tensors; ++t)   // every tensor is checked before anything is enqueued
    if (!W[t] || d_out[t] <= 0 || d_in[t] <= 0) return GIFT_ERR_INVALID_ARG;
  if (scaling != GIFT_SCALE_TENSOR) {   // the block scalings need no amax pass
    for (int t = 0; t < n_tensors; ++t) {
      const gift_status st = gift_boundary_hit_rate(ctx, W[t], d_out[t], d_in[t], fmt, scaling, d_counts + 3 * t,
                                                    ws, ws_bytes, d_status, stream);
      if (st != GIFT_OK) return st;
    }
    return GIFT_OK;
  }
  const CodecWs need = codec_layout(nullptr, ctx->sms, GIFT_OP_AMAX, GIFT_XF_IDENTITY, 1, 1);
  if (!ws || ws_bytes < need.bytes) return GIFT_ERR_INVALID_ARG;
  const CodecWs w = codec_layout(ws, ctx->sms, GIFT_OP_AMAX, GIFT_XF_IDENTITY, 1, 1);
  const Launch L = mk(ctx, d_status, stream);
  for (int t0 = 0; t0 < n_tensors; t0 += kMaxReplicas) {   // the 64 amax words of the workspace
    const int m = (n_tensors - t0 < kMaxReplicas) ? n_tensors - t0 : kMaxReplicas;
    HitsArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int t = 0; t < m; ++t) {
      a.x[t] = W[t0 + t];
      a.n[t] = (size_t)d_out[t0 + t] * d_in[t0 + t];
    }
    CK(launch_hits_multi(L, fmt, a, m, reinterpret_cast<uint32_t *>(w.amax), d_counts + 3 * (size_t)t0));
  }
  return GIFT_OK;
}

// Fragile-layer selection from a profiling window (host only).  Scores are formed in double
// from the integer counts, so every comparison below is exact and repeatable.
gift_status gift_select_fragile(int L, const unsigned long long *counts, int k, int k_min, int k_max, int *order,
                                double *scores, int *k_out) {
  if (L < 1 || !counts || !order || !k_out || k < 0 || k > L) return GIFT_ERR_INVALID_ARG;
  if (k == 0 && !(1 <= k_min && k_min <= k_max && k_max <= L)) return GIFT_ERR_INVALID_ARG;
  std::vector<double> s(L);
  for (int l = 0; l < L; ++l) {
    const unsigned long long up = counts[3 * (size_t)l], lo = counts[3 * (size_t)l + 1],
                             n = counts[3 * (size_t)l + 2];
    if (up > n || lo > n) return GIFT_ERR_INVALID_ARG;   // not the counts of one layer
    s[l] = n ? (double)(up + lo) / (double)n : 0.0;
  }
  std::vector<int> o(L);
  std::iota(o.begin(), o.end(), 0);
  std::sort(o.begin(), o.end(), [&](int a, int b) { return s[a] > s[b] || (s[a] == s[b] && a < b); });
  if (k == 0) {
    k = k_min;
    if (k_min < L) {
      // the largest drop between consecutive ranked scores; equal drops keep the smaller k
      const int hi = std::min(k_max, L - 1);
      double best = s[o[k_min - 1]] - s[o[k_min]];
      for (int c = k_min + 1; c <= hi; ++c) {
        const double drop = s[o[c - 1]] - s[o[c]];
        if (drop > best) {
          best = drop;
          k = c;
        }
      }
    }
  }
  for (int i = 0; i < L; ++i) order[i] = o[i];
  if (scores)
    for (int l = 0; l < L; ++l) scores[l] = s[l];
  *k_out = k;
  return GIFT_OK;
}

}  // extern "C"
