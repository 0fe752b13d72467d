// CPU oracle of the GIFT per-layer gradient codec in plain C++17.  TEST INFRASTRUCTURE ONLY.
//
// This file states, slowly and plainly, what the codec computes.  It is used by the tests,
// by the smoke check and by the benchmark's CPU-baseline leg, through the ctypes wrapper
// oracle/cpp.py; the product (the CUDA library and its binding) never loads it, and it
// shares no code, header, table or constant with the CUDA kernels.  It is the second
// statement of the oracle beside oracle/gift_oracle.py (numpy): both are pinned by the same
// tests, and they must agree.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off (no fused multiply-add anywhere, so every FP32
// operation written here is one IEEE round-to-nearest-even operation).  Without -fopenmp it
// is single-threaded.  With -fopenmp the `omp parallel for` loops split independent output
// elements across threads; every element is still computed by one thread in the same order,
// so the results are identical to the single-threaded build.
//
// Sources, cited by page title and section (the pages give equations and an algorithm, no
// code):
//   [notes]    "GIFT 阅读笔记:量化用的坐标系,比量化器本身更重要" (GIFT reading notes,
//              zhongzhuzhou.org).  Sections: 前置知识 (prerequisites: "What FP8 is",
//              data-parallel averaging eq. (1), K-FAC eqs. (2)-(4)), 核心想法 (core idea,
//              steps 1-3, eqs. (5)-(14)), 三次简化 (three simplifications, eqs. (15)-(17)
//              and the profiling procedure), 算法 1 (Algorithm 1), 玩具例子 (the worked 2x2
//              example).
//   [abstract] "GIFT: Geometry-Informed Low-precision Gradient Communication for LLM
//              Pretraining" (shd-paper.top summary): FP8 and NVFP4 formats.
//
// Readings where the pages are silent (the same as the numpy oracle's):
//   * rounding to FP8/FP4 is round-to-nearest-even with saturation to the largest finite
//     value; the sign of zero is kept;
//   * s = amax / FMAX is stored and elements are scaled by m = FMAX / amax, both single FP32
//     divisions; amax = 0 gives s = m = 0; an m beyond FP32 is clamped to the largest finite;
//   * the rank-r factor is completed with sigma I, sigma the mean of the eigenvalues of A
//     outside the top r (trace preserved); r = d_in gives sigma = 1;
//   * NVFP4 = E2M1 codes, one E4M3 scale per 16 consecutive elements of a row, one FP32
//     tensor scale s_t = amax / 2688;
//   * the replica reduce dequantises each replica with its own scale, then averages in
//     replica order.
//
// Every function is pinned by tests/test_oracle_pins.py (parity pinned).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---- number formats ([notes] prerequisites "What FP8 is"; [abstract] NVFP4) ----------

struct Format {
  int ebits, mbits, bias;
  double maxval;
  int nbits;
  int emin() const { return 1 - bias; }
  double min_subnormal() const { return std::ldexp(1.0, emin() - mbits); }
};

// 0 = E4M3 (largest finite 448, no infinities), 1 = E5M2 (largest finite 57344),
// 2 = E2M1 (the NVFP4 element format, largest 6)
const Format kFormats[3] = {{4, 3, 7, 448.0, 8}, {5, 2, 15, 57344.0, 8}, {2, 1, 1, 6.0, 4}};

const float kF32Max = std::numeric_limits<float>::max();

// Nearest value of the format to the exact value of y (ties to even), saturating at the
// largest finite value; NaN stays NaN.  The quantum of a binade is a power of two, so a / q
// is exact and rint (round half to even in the default mode) does the rounding.
double round_to_format(float y, const Format &f) {
  const double yd = static_cast<double>(y);
  if (std::isnan(yd)) return yd;
  const double a = std::fabs(yd);
  double v;
  if (a >= f.maxval) {
    v = f.maxval;
  } else {
    int ex = 0;
    std::frexp(a, &ex);                       // a = frac * 2^ex, frac in [0.5, 1)
    int e = ex - 1;                           // binade exponent
    if (e < f.emin()) e = f.emin();           // subnormal range has the smallest normal's quantum
    const double q = std::ldexp(1.0, e - f.mbits);
    v = std::nearbyint(a / q) * q;
    if (v > f.maxval) v = f.maxval;
  }
  return std::copysign(v, yd);
}

// Bit pattern of an exactly representable value v of the format.
uint8_t value_to_code(double v, const Format &f) {
  if (std::isnan(v)) return f.ebits == 2 ? 0 : static_cast<uint8_t>((1 << (f.nbits - 1)) - 1);
  const unsigned sign = std::signbit(v) ? 1u : 0u;
  const double a = std::fabs(v);
  unsigned e_field = 0, mant = 0;
  if (a != 0.0) {
    if (a >= std::ldexp(1.0, f.emin())) {
      int ex = 0;
      std::frexp(a, &ex);
      const int e = ex - 1;
      e_field = static_cast<unsigned>(e + f.bias);
      mant = static_cast<unsigned>(a / std::ldexp(1.0, e - f.mbits) - std::ldexp(1.0, f.mbits));
    } else {
      mant = static_cast<unsigned>(a / f.min_subnormal());
    }
  }
  return static_cast<uint8_t>((sign << (f.nbits - 1)) | (e_field << f.mbits) | mant);
}

uint8_t encode1(float y, const Format &f) { return value_to_code(round_to_format(y, f), f); }

// Exact value of a code from its sign, exponent and mantissa fields.
double decode1(uint8_t code, int fmt) {
  const Format &f = kFormats[fmt];
  const unsigned c = code & ((1u << f.nbits) - 1);
  const double sign = ((c >> (f.nbits - 1)) & 1) ? -1.0 : 1.0;
  const unsigned e_field = (c >> f.mbits) & ((1u << f.ebits) - 1);
  const unsigned mant = c & ((1u << f.mbits) - 1);
  const unsigned mag = c & ((1u << (f.nbits - 1)) - 1);
  if (fmt == 0 && mag == 0x7F) return std::numeric_limits<double>::quiet_NaN();
  if (fmt == 1 && mag == 0x7C) return sign * std::numeric_limits<double>::infinity();
  if (fmt == 1 && mag > 0x7C) return std::numeric_limits<double>::quiet_NaN();
  if (e_field == 0) return sign * mant * f.min_subnormal();
  return sign * (1.0 + mant / std::ldexp(1.0, f.mbits)) * std::ldexp(1.0, static_cast<int>(e_field) - f.bias);
}

// ---- scaling ([notes] prerequisites "What FP8 is": s = amax / FP8_MAX) ----------------

// amax = max |x| over n elements; false on a NaN or infinity.
bool abs_max(const float *x, int64_t n, float *amax) {
  float m = 0.0f;
  bool finite = true;
#pragma omp parallel for reduction(max : m) reduction(&& : finite)
  for (int64_t i = 0; i < n; ++i) {
    if (!std::isfinite(x[i])) finite = false;
    const float a = std::fabs(x[i]);
    if (a > m) m = a;
  }
  *amax = m;
  return finite;
}

void scale_pair(float amax, const Format &f, float *s, float *m) {
  if (amax == 0.0f) {
    *s = 0.0f;
    *m = 0.0f;
    return;
  }
  const float fmax = static_cast<float>(f.maxval);
  *s = amax / fmax;
  float mm = fmax / amax;
  if (std::isinf(mm)) mm = kF32Max;
  *m = mm;
}

// code = RNE_satfinite(fl32(x * m))
void quantize_with_multiplier(const float *x, int64_t n, float m, const Format &f, uint8_t *codes) {
#pragma omp parallel for
  for (int64_t i = 0; i < n; ++i) {
    const float y = x[i] * m;
    codes[i] = encode1(y, f);
  }
}

// x_hat = fl32(value(code) * s)
void dequantize(const uint8_t *codes, int64_t n, float s, int fmt, float *out) {
#pragma omp parallel for
  for (int64_t i = 0; i < n; ++i) {
    const float v = static_cast<float>(decode1(codes[i], fmt));
    out[i] = v * s;
  }
}

// ---- dense double helpers (plain loops) ------------------------------------------------

// C (m x n) = A (m x k) * B (k x n), row-major, double.
void matmul(const double *A, const double *B, int64_t m, int64_t k, int64_t n, double *C) {
#pragma omp parallel for
  for (int64_t i = 0; i < m; ++i) {
    double *c = C + i * n;
    for (int64_t j = 0; j < n; ++j) c[j] = 0.0;
    for (int64_t p = 0; p < k; ++p) {
      const double a = A[i * k + p];
      const double *b = B + p * n;
      for (int64_t j = 0; j < n; ++j) c[j] += a * b[j];
    }
  }
}

// C (m x n) = A (m x k) * B^T with B n x k.
void matmul_bt(const double *A, const double *B, int64_t m, int64_t k, int64_t n, double *C) {
#pragma omp parallel for
  for (int64_t i = 0; i < m; ++i)
    for (int64_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int64_t p = 0; p < k; ++p) acc += A[i * k + p] * B[j * k + p];
      C[i * n + j] = acc;
    }
}

// C (m x n) = A^T B with A k x m, B k x n.
void matmul_at(const double *A, const double *B, int64_t k, int64_t m, int64_t n, double *C) {
#pragma omp parallel for
  for (int64_t i = 0; i < m; ++i) {
    double *c = C + i * n;
    for (int64_t j = 0; j < n; ++j) c[j] = 0.0;
    for (int64_t p = 0; p < k; ++p) {
      const double a = A[p * m + i];
      const double *b = B + p * n;
      for (int64_t j = 0; j < n; ++j) c[j] += a * b[j];
    }
  }
}

// Thin Q (n x k, n >= k) of X = Q R by Householder reflections (Golub & Van Loan, "Matrix
// Computations", section 5.2: reflector v = x + sign(x_1) |x| e_1, so R's diagonal is
// -sign(x_1) |x|), Q formed by applying the reflectors to the first k columns of I.
void householder_q(const double *X, int64_t n, int64_t k, double *Q) {
  std::vector<double> R(X, X + n * k);
  std::vector<double> V(static_cast<size_t>(n * k), 0.0), beta(static_cast<size_t>(k), 0.0);
  for (int64_t j = 0; j < k; ++j) {
    double norm2 = 0.0;
    for (int64_t i = j; i < n; ++i) norm2 += R[i * k + j] * R[i * k + j];
    const double norm = std::sqrt(norm2);
    if (norm == 0.0) {
      beta[j] = 0.0;
      continue;
    }
    const double x1 = R[j * k + j];
    const double alpha = (x1 >= 0.0) ? -norm : norm;   // R_jj
    double vnorm2 = 0.0;
    for (int64_t i = j; i < n; ++i) {
      const double vi = (i == j) ? x1 - alpha : R[i * k + j];
      V[i * k + j] = vi;
      vnorm2 += vi * vi;
    }
    beta[j] = (vnorm2 > 0.0) ? 2.0 / vnorm2 : 0.0;
    // R <- (I - beta v v^T) R on columns j..k-1
    for (int64_t c = j; c < k; ++c) {
      double dot = 0.0;
      for (int64_t i = j; i < n; ++i) dot += V[i * k + j] * R[i * k + c];
      const double t = beta[j] * dot;
      for (int64_t i = j; i < n; ++i) R[i * k + c] -= t * V[i * k + j];
    }
  }
  // Q = H_0 H_1 ... H_{k-1} I[:, :k], applied last reflector first
  for (int64_t i = 0; i < n; ++i)
    for (int64_t c = 0; c < k; ++c) Q[i * k + c] = (i == c) ? 1.0 : 0.0;
  for (int64_t j = k - 1; j >= 0; --j) {
    if (beta[j] == 0.0) continue;
    for (int64_t c = 0; c < k; ++c) {
      double dot = 0.0;
      for (int64_t i = j; i < n; ++i) dot += V[i * k + j] * Q[i * k + c];
      const double t = beta[j] * dot;
      for (int64_t i = j; i < n; ++i) Q[i * k + c] -= t * V[i * k + j];
    }
  }
}

}  // namespace

extern "C" {

// ---- formats -----------------------------------------------------------------------------

// Constants of a format: ebits, mbits, bias, nbits and the largest finite value.
void or_format_info(int fmt, int *ebits, int *mbits, int *bias, int *nbits, double *maxval) {
  const Format &f = kFormats[fmt];
  *ebits = f.ebits;
  *mbits = f.mbits;
  *bias = f.bias;
  *nbits = f.nbits;
  *maxval = f.maxval;
}

void or_encode(const float *y, int64_t n, int fmt, uint8_t *codes) {
  const Format &f = kFormats[fmt];
#pragma omp parallel for
  for (int64_t i = 0; i < n; ++i) codes[i] = encode1(y[i], f);
}

void or_decode(const uint8_t *codes, int64_t n, int fmt, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = decode1(codes[i], fmt);
}

// ---- scaling and FP8 quantisation (Algorithm 1: Scale, Q, Dequantize) -----------------

// Returns 1 (non-finite) or 0.
int or_abs_max(const float *x, int64_t n, float *amax) { return abs_max(x, n, amax) ? 0 : 1; }

void or_scale_pair(float amax, int fmt, float *s, float *m) { scale_pair(amax, kFormats[fmt], s, m); }

void or_quantize_with_multiplier(const float *x, int64_t n, float m, int fmt, uint8_t *codes) {
  quantize_with_multiplier(x, n, m, kFormats[fmt], codes);
}

void or_dequantize(const uint8_t *codes, int64_t n, float s, int fmt, float *out) {
  dequantize(codes, n, s, fmt, out);
}

// Per-tensor scaling: the tensor's own amax, or amax_in (the AllReduceMax'd shared scale).
// Returns 1 on a non-finite element (nothing else written), else 0.
int or_quantize_tensor(const float *x, int64_t n, int fmt, const float *amax_in, uint8_t *codes, float *s,
                       float *amax_used) {
  float local = 0.0f;
  if (!abs_max(x, n, &local)) return 1;
  const float a = amax_in ? *amax_in : local;
  float m = 0.0f;
  scale_pair(a, kFormats[fmt], s, &m);
  quantize_with_multiplier(x, n, m, kFormats[fmt], codes);
  *amax_used = a;
  return 0;
}

// amax of every b x b tile of a d_out x d_in tensor (edge tiles clipped),
// am[ceil(d_out/b)][ceil(d_in/b)].  Returns 1 on a non-finite element.
int or_block_amax(const float *x, int d_out, int d_in, int b, float *am) {
  const int nbr = (d_out + b - 1) / b, nbc = (d_in + b - 1) / b;
  bool finite = true;
  for (int bi = 0; bi < nbr; ++bi)
    for (int bj = 0; bj < nbc; ++bj) {
      float m = 0.0f;
      for (int i = bi * b; i < d_out && i < (bi + 1) * b; ++i)
        for (int j = bj * b; j < d_in && j < (bj + 1) * b; ++j) {
          const float v = x[(int64_t)i * d_in + j];
          if (!std::isfinite(v)) finite = false;
          if (std::fabs(v) > m) m = std::fabs(v);
        }
      am[bi * nbc + bj] = m;
    }
  return finite ? 0 : 1;
}

// Per-block scaling on b x b tiles ([notes] prerequisites: per-block scales; b = 128 for the
// codec).  amax_in (nullable) overrides the blocks' own amax.
int or_quantize_block2d(const float *x, int d_out, int d_in, int b, int fmt, const float *amax_in, uint8_t *codes,
                        float *scales, float *am) {
  const int nbr = (d_out + b - 1) / b, nbc = (d_in + b - 1) / b;
  if (amax_in) {
    std::memcpy(am, amax_in, sizeof(float) * nbr * nbc);
  } else if (or_block_amax(x, d_out, d_in, b, am)) {
    return 1;
  }
  const Format &f = kFormats[fmt];
  for (int bi = 0; bi < nbr; ++bi)
    for (int bj = 0; bj < nbc; ++bj) {
      float s = 0.0f, m = 0.0f;
      scale_pair(am[bi * nbc + bj], f, &s, &m);
      scales[bi * nbc + bj] = s;
      for (int i = bi * b; i < d_out && i < (bi + 1) * b; ++i)
        for (int j = bj * b; j < d_in && j < (bj + 1) * b; ++j) {
          const int64_t k = (int64_t)i * d_in + j;
          const float y = x[k] * m;
          codes[k] = encode1(y, f);
        }
    }
  return 0;
}

void or_dequantize_block2d(const uint8_t *codes, int d_out, int d_in, int b, const float *scales, int fmt,
                           float *out) {
  const int nbc = (d_in + b - 1) / b;
  for (int i = 0; i < d_out; ++i)
    for (int j = 0; j < d_in; ++j) {
      const int64_t k = (int64_t)i * d_in + j;
      const float v = static_cast<float>(decode1(codes[k], fmt));
      out[k] = v * scales[(i / b) * nbc + j / b];
    }
}

// 1-D blocks of b consecutive elements of the flattened tensor (the experiments' per-block
// Euclidean baseline, b = 512), the last block shorter.  amax_in: one value per block.
int or_quantize_block1d(const float *x, int64_t n, int b, int fmt, const float *amax_in, uint8_t *codes,
                        float *scales, float *am) {
  const int64_t nb = (n + b - 1) / b;
  const Format &f = kFormats[fmt];
  for (int64_t i = 0; i < nb; ++i) {
    const int64_t lo = i * b, hi = (lo + b < n) ? lo + b : n;
    float a = 0.0f;
    if (amax_in) {
      a = amax_in[i];
    } else if (!abs_max(x + lo, hi - lo, &a)) {
      return 1;
    }
    am[i] = a;
    float s = 0.0f, m = 0.0f;
    scale_pair(a, f, &s, &m);
    scales[i] = s;
    quantize_with_multiplier(x + lo, hi - lo, m, f, codes + lo);
  }
  return 0;
}

void or_dequantize_block1d(const uint8_t *codes, int64_t n, int b, const float *scales, int fmt, float *out) {
  for (int64_t i = 0; i < n; ++i) {
    const float v = static_cast<float>(decode1(codes[i], fmt));
    out[i] = v * scales[i / b];
  }
}

// ---- NVFP4 ([abstract]: FP8 and NVFP4) ---------------------------------------------------

// packed[d_out][d_in/2] (even column in the low nibble), block_scales[d_out][d_in/16] E4M3
// bytes, *s_t the FP32 tensor scale, *at the tensor amax used.  For each group of 16:
// e_b = E4M3(a_b / fl32(6 s_t)), eff = fl32(e_b s_t), r_b = 1 / eff (0 when eff = 0, the
// largest finite FP32 when it overflows), code = E2M1(fl32(x r_b)).
// Returns 1 on a non-finite element, 2 when d_in is not a multiple of 16.
int or_quantize_nvfp4(const float *x, int d_out, int d_in, const float *amax_in, uint8_t *packed,
                      uint8_t *block_scales, float *s_t_out, float *at_out) {
  if (d_in % 16) return 2;
  float local = 0.0f;
  if (!abs_max(x, (int64_t)d_out * d_in, &local)) return 1;
  const float at = amax_in ? *amax_in : local;
  const float s_t = at / 2688.0f;   // 448 * 6, exact in FP32
  const float six_st = 6.0f * s_t;
  const Format &e4 = kFormats[0], &e2 = kFormats[2];
  const int groups = d_in / 16;
#pragma omp parallel for
  for (int i = 0; i < d_out; ++i) {
    for (int g = 0; g < groups; ++g) {
      const float *xg = x + (int64_t)i * d_in + g * 16;
      float ab = 0.0f;
      for (int t = 0; t < 16; ++t)
        if (std::fabs(xg[t]) > ab) ab = std::fabs(xg[t]);
      const float ratio = (s_t == 0.0f) ? 0.0f : ab / six_st;
      const uint8_t eb_code = encode1(ratio, e4);
      const float eb = static_cast<float>(decode1(eb_code, 0));
      const float eff = eb * s_t;
      float rb = (eff == 0.0f) ? 0.0f : 1.0f / eff;
      if (std::isinf(rb)) rb = kF32Max;
      block_scales[(int64_t)i * groups + g] = eb_code;
      for (int t = 0; t < 16; t += 2) {
        const float y0 = xg[t] * rb, y1 = xg[t + 1] * rb;
        const uint8_t c0 = encode1(y0, e2) & 0xF, c1 = encode1(y1, e2) & 0xF;
        packed[(int64_t)i * (d_in / 2) + (g * 16 + t) / 2] = static_cast<uint8_t>(c0 | (c1 << 4));
      }
    }
  }
  *s_t_out = s_t;
  *at_out = at;
  return 0;
}

// x_hat = fl32(fl32(value(code) * value(e_b)) * s_t)
void or_dequantize_nvfp4(const uint8_t *packed, const uint8_t *block_scales, float s_t, int d_out, int d_in,
                         float *out) {
  const int groups = d_in / 16;
  for (int i = 0; i < d_out; ++i)
    for (int j = 0; j < d_in; ++j) {
      const uint8_t byte = packed[(int64_t)i * (d_in / 2) + j / 2];
      const uint8_t c = (j % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      const float v = static_cast<float>(decode1(c, 2));
      const float eb = static_cast<float>(decode1(block_scales[(int64_t)i * groups + j / 16], 0));
      const float p = v * eb;
      out[(int64_t)i * d_in + j] = p * s_t;
    }
}

// ---- replica reduce ([notes] eq. (1); Algorithm 1: AllReduceSum, Dequantize, / N) ------

// out = (deq_0 + deq_1 + ... + deq_{R-1}) / R: FP32 additions left to right, starting from
// replica 0's values.  deq holds the R dequantised replicas back to back (R x n).
void or_replica_mean(const float *deq, int R, int64_t n, float *out) {
  const float Rf = static_cast<float>(R);
#pragma omp parallel for
  for (int64_t i = 0; i < n; ++i) {
    float acc = deq[i];
    for (int r = 1; r < R; ++r) acc = acc + deq[(int64_t)r * n + i];
    out[i] = acc / Rf;
  }
}

// ---- boundary-hit profiler ([notes] simplification 3) ----------------------------------

// counts[0] = #{|code| is the largest finite code}, counts[1] = #{x != 0 and |code| = 0},
// counts[2] = n, for codes of x quantised with its own scale.
void or_boundary_counts(const float *x, const uint8_t *codes, int64_t n, int fmt, uint64_t *counts) {
  const uint8_t maxc = encode1(static_cast<float>(kFormats[fmt].maxval), kFormats[fmt]);
  uint64_t up = 0, lo = 0;
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t mag = codes[i] & 0x7F;
    if (mag == maxc) ++up;
    if (x[i] != 0.0f && mag == 0) ++lo;
  }
  counts[0] = up;
  counts[1] = lo;
  counts[2] = static_cast<uint64_t>(n);
}

// (upper + lower) / n per layer over a window (counts: L x 3), 0 when n = 0.
void or_window_scores(const uint64_t *counts, int L, double *scores) {
  for (int l = 0; l < L; ++l) {
    const uint64_t *c = counts + 3 * l;
    scores[l] = c[2] ? static_cast<double>(c[0] + c[1]) / static_cast<double>(c[2]) : 0.0;
  }
}

// Layer indices by descending score, ties to the lower index (insertion sort, stable).
void or_rank_layers(const double *scores, int L, int *order) {
  for (int i = 0; i < L; ++i) order[i] = i;
  for (int i = 1; i < L; ++i) {
    const int v = order[i];
    int j = i - 1;
    while (j >= 0 && scores[order[j]] < scores[v]) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }
}

// The k in [k_min, min(k_max, L - 1)] with the largest drop ranked[k-1] - ranked[k]
// (equal drops: the smaller k); L when k_min == L.  -1 on bad bounds.
int or_knee_count(const double *ranked, int L, int k_min, int k_max) {
  if (!(1 <= k_min && k_min <= k_max && k_max <= L)) return -1;
  if (k_min == L) return L;
  const int hi = (k_max < L - 1) ? k_max : L - 1;
  int best_k = k_min;
  double best = 0.0;
  bool have = false;
  for (int k = k_min; k <= hi; ++k) {
    const double drop = ranked[k - 1] - ranked[k];
    if (!have || drop > best) {
      best_k = k;
      best = drop;
      have = true;
    }
  }
  return best_k;
}

// ---- K-FAC factors ([notes] prerequisites "K-FAC", eq. (4): A = E[a a^T]) --------------

// A (d x d) = a^T a / T in double, a: T x d (inputs widened exactly by the caller).
void or_kfac_factor(const double *a, int64_t T, int64_t d, double *A) {
  matmul_at(a, a, T, d, d, A);
  const double Td = static_cast<double>(T);
  for (int64_t i = 0; i < d * d; ++i) A[i] /= Td;
}

// tr(A) of an n x n matrix.
double or_trace(const double *A, int64_t n) {
  double t = 0.0;
  for (int64_t i = 0; i < n; ++i) t += A[i * n + i];
  return t;
}

// tr(a^T a / T) = (sum of the squares of the activations) / T, without forming A.
double or_activation_trace(const double *a, int64_t T, int64_t d) {
  double t = 0.0;
  for (int64_t i = 0; i < T * d; ++i) t += a[i] * a[i];
  return t / static_cast<double>(T);
}

// Textbook Cholesky A = L L^T ([notes] core idea step 2, eq. (7)), column by column.
// Returns -1 on success, else the index of the first non-positive pivot.
int or_cholesky(const double *A, int64_t n, double *L) {
  for (int64_t i = 0; i < n * n; ++i) L[i] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double d = A[j * n + j];
    for (int64_t p = 0; p < j; ++p) d -= L[j * n + p] * L[j * n + p];
    if (!(d > 0.0)) return static_cast<int>(j);
    const double ljj = std::sqrt(d);
    L[j * n + j] = ljj;
#pragma omp parallel for
    for (int64_t i = j + 1; i < n; ++i) {
      double s = A[i * n + j];
      for (int64_t p = 0; p < j; ++p) s -= L[i * n + p] * L[j * n + p];
      L[i * n + j] = s / ljj;
    }
  }
  return -1;
}

// X = L^-1 of a lower-triangular L by forward substitution, row by row of L X = I.
void or_lower_inverse(const double *L, int64_t n, double *X) {
  for (int64_t i = 0; i < n * n; ++i) X[i] = 0.0;
  for (int64_t i = 0; i < n; ++i) {
#pragma omp parallel for
    for (int64_t c = 0; c <= i; ++c) {
      double rhs = (c == i) ? 1.0 : 0.0;
      for (int64_t p = c; p < i; ++p) rhs -= L[i * n + p] * X[p * n + c];
      X[i * n + c] = rhs / L[i * n + i];
    }
  }
}

// X (m x n) with X L^T = W (X = W L^-T), forward substitution over the columns of X.
void or_solve_right_lower_t(const double *W, const double *L, int64_t m, int64_t n, double *X) {
#pragma omp parallel for
  for (int64_t r = 0; r < m; ++r)
    for (int64_t j = 0; j < n; ++j) {
      double s = W[r * n + j];
      for (int64_t p = 0; p < j; ++p) s -= X[r * n + p] * L[j * n + p];
      X[r * n + j] = s / L[j * n + j];
    }
}

// Y (m x n) with L Y = W (Y = L^-1 W), L m x m, forward substitution over the rows of Y.
void or_solve_left_lower(const double *L, const double *W, int64_t m, int64_t n, double *Y) {
  for (int64_t i = 0; i < m; ++i) {
#pragma omp parallel for
    for (int64_t c = 0; c < n; ++c) {
      double s = W[i * n + c];
      for (int64_t p = 0; p < i; ++p) s -= L[i * m + p] * Y[p * n + c];
      Y[i * n + c] = s / L[i * m + i];
    }
  }
}

void or_matmul(const double *A, const double *B, int64_t m, int64_t k, int64_t n, double *C) {
  matmul(A, B, m, k, n, C);
}

void or_matmul_bt(const double *A, const double *B, int64_t m, int64_t k, int64_t n, double *C) {
  matmul_bt(A, B, m, k, n, C);
}

// ---- symmetric eigensolver -------------------------------------------------------------

// Cyclic Jacobi eigendecomposition of a symmetric n x n matrix in double: each rotation
// zeroes one off-diagonal pair (p, q) with the smaller rotation angle (Golub & Van Loan,
// "Matrix Computations", section 8.5), sweeps until the off-diagonal norm is below tol times
// the matrix norm.  w: eigenvalues in descending order (stable), V: eigenvectors as columns.
// Returns the number of sweeps taken.
int or_jacobi_eigh(const double *S, int64_t n, double tol, int max_sweeps, double *w, double *V) {
  std::vector<double> A(S, S + n * n), Vt(static_cast<size_t>(n * n), 0.0);
  for (int64_t i = 0; i < n; ++i) Vt[i * n + i] = 1.0;
  int sweeps = 0;
  for (; sweeps < max_sweeps; ++sweeps) {
    double off = 0.0, all = 0.0;
    for (int64_t i = 0; i < n; ++i)
      for (int64_t j = 0; j < n; ++j) {
        all += A[i * n + j] * A[i * n + j];
        if (j < i) off += A[i * n + j] * A[i * n + j];
      }
    const double scale = std::sqrt(all) > 1e-300 ? std::sqrt(all) : 1e-300;
    if (std::sqrt(off) <= tol * scale) break;
    for (int64_t p = 0; p < n - 1; ++p)
      for (int64_t q = p + 1; q < n; ++q) {
        const double apq = A[p * n + q];
        if (apq == 0.0 || std::fabs(apq) <= 1e-18 * std::sqrt(std::fabs(A[p * n + p] * A[q * n + q]))) continue;
        const double theta = (A[q * n + q] - A[p * n + p]) / (2.0 * apq);
        double t = 1.0;
        if (theta != 0.0) t = (theta > 0 ? 1.0 : -1.0) / (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0), s = t * c;
        for (int64_t i = 0; i < n; ++i) {   // columns p, q: A <- A J
          const double ap = A[i * n + p], aq = A[i * n + q];
          A[i * n + p] = c * ap - s * aq;
          A[i * n + q] = s * ap + c * aq;
        }
        for (int64_t j = 0; j < n; ++j) {   // rows p, q: A <- J^T A
          const double ap = A[p * n + j], aq = A[q * n + j];
          A[p * n + j] = c * ap - s * aq;
          A[q * n + j] = s * ap + c * aq;
        }
        A[p * n + q] = A[q * n + p] = 0.0;
        for (int64_t i = 0; i < n; ++i) {   // V <- V J
          const double vp = Vt[i * n + p], vq = Vt[i * n + q];
          Vt[i * n + p] = c * vp - s * vq;
          Vt[i * n + q] = s * vp + c * vq;
        }
      }
  }
  std::vector<int64_t> order(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) order[i] = i;
  for (int64_t i = 1; i < n; ++i) {   // stable insertion sort by descending eigenvalue
    const int64_t v = order[i];
    int64_t j = i - 1;
    while (j >= 0 && A[order[j] * n + order[j]] < A[v * n + v]) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }
  for (int64_t c = 0; c < n; ++c) {
    w[c] = A[order[c] * n + order[c]];
    for (int64_t i = 0; i < n; ++i) V[i * n + c] = Vt[i * n + order[c]];
  }
  return sweeps;
}

// Y (n x k) = A X for the operator of a subspace iteration: mode 0, M is an explicit n x n
// matrix A; mode 1, M holds T x n activations and A X = a^T (a X) / T (A never formed);
// mode 2, the caller's callback.
typedef void (*or_apply_fn)(const double *X, int64_t n, int64_t k, double *Y, void *user);

static void apply_op(int mode, const double *M, int64_t T, int64_t n, int64_t k, const double *X, double *Y,
                     or_apply_fn cb, void *user) {
  if (mode == 0) {
    matmul(M, X, n, n, k, Y);
  } else if (mode == 1) {
    std::vector<double> Z(static_cast<size_t>(T * k));
    matmul(M, X, T, n, k, Z.data());
    matmul_at(M, Z.data(), T, n, k, Y);
    const double Td = static_cast<double>(T);
    for (int64_t i = 0; i < n * k; ++i) Y[i] /= Td;
  } else {
    cb(X, n, k, Y, user);
  }
}

// Top-k Ritz pairs of a symmetric PSD operator by block subspace iteration ([notes]
// simplification 2, eq. (17), the rank-r approximation; N. Halko, P.-G. Martinsson, J. Tropp,
// "Finding structure with randomness", SIAM Review 2011, Alg. 4.4 with Rayleigh-Ritz):
// Q_0 = orth(Omega) with the caller's Gaussian start Omega (n x k); Q_{i+1} = orth(A Q_i)
// for `iters` steps; B = Q^T A Q symmetrised; Jacobi eigenpairs (mu, V) of B; U = Q V.
// mu: k values descending; U: n x k.
void or_subspace_iteration(int mode, const double *M, int64_t T, int64_t n, int64_t k, int iters,
                           const double *omega, or_apply_fn cb, void *user, double *mu, double *U) {
  std::vector<double> Q(static_cast<size_t>(n * k)), Y(static_cast<size_t>(n * k));
  householder_q(omega, n, k, Q.data());
  for (int it = 0; it < iters; ++it) {
    apply_op(mode, M, T, n, k, Q.data(), Y.data(), cb, user);
    householder_q(Y.data(), n, k, Q.data());
  }
  apply_op(mode, M, T, n, k, Q.data(), Y.data(), cb, user);
  std::vector<double> B(static_cast<size_t>(k * k)), Bs(static_cast<size_t>(k * k)), V(static_cast<size_t>(k * k));
  matmul_at(Q.data(), Y.data(), n, k, k, B.data());
  for (int64_t i = 0; i < k; ++i)
    for (int64_t j = 0; j < k; ++j) Bs[i * k + j] = 0.5 * (B[i * k + j] + B[j * k + i]);
  or_jacobi_eigh(Bs.data(), k, 1e-15, 40, mu, V.data());
  matmul(Q.data(), V.data(), n, k, k, U);
}

// ---- the rank-r factor and its transform ([notes] simplification 2, eq. (17)) ----------

// From the top eigenpairs (mu_all descending, V_all n x k columns) and tr(A): U = V[:, :r],
// mu = mu_all[:r], sigma = (tr A - sum mu) / (d - r) (1 when r = d).  Returns 1 when sigma or
// a mu is not positive.
int or_lowrank_from_eigs(const double *mu_all, const double *V_all, int64_t k, double trace, int64_t d, int64_t r,
                         double *U, double *mu, double *sigma) {
  double sum = 0.0;
  for (int64_t i = 0; i < r; ++i) {
    mu[i] = mu_all[i];
    sum += mu_all[i];
  }
  for (int64_t i = 0; i < d; ++i)
    for (int64_t c = 0; c < r; ++c) U[i * r + c] = V_all[i * k + c];
  const double s = (r == d) ? 1.0 : (trace - sum) / static_cast<double>(d - r);
  *sigma = s;
  bool ok = s > 0.0;
  for (int64_t i = 0; i < r; ++i) ok = ok && mu[i] > 0.0;
  return ok ? 0 : 1;
}

// c_i = mu_i^-1/2 - sigma^-1/2 (whitening) or mu_i^1/2 - sigma^1/2 (map back).
static void lowrank_coeffs(const double *mu, int64_t r, double sigma, int inverse, double *c) {
  for (int64_t i = 0; i < r; ++i)
    c[i] = inverse ? std::sqrt(mu[i]) - std::sqrt(sigma) : 1.0 / std::sqrt(mu[i]) - 1.0 / std::sqrt(sigma);
}

// W~ = W T_A = sigma^-1/2 W + ((W U) diag(c)) U^T (inverse = 0), or the map back
// W^ = X T_A^-1 = sigma^1/2 X + ((X U) diag(c')) U^T (inverse = 1).  W: m x d, U: d x r.
void or_lowrank_apply(const double *W, int64_t m, int64_t d, const double *U, const double *mu, int64_t r,
                      double sigma, int inverse, double *out) {
  std::vector<double> c(static_cast<size_t>(r)), P(static_cast<size_t>(m * r));
  lowrank_coeffs(mu, r, sigma, inverse, c.data());
  matmul(W, U, m, d, r, P.data());
  for (int64_t i = 0; i < m; ++i)
    for (int64_t j = 0; j < r; ++j) P[i * r + j] *= c[j];
  matmul_bt(P.data(), U, m, r, d, out);
  const double root = std::sqrt(sigma);
  for (int64_t i = 0; i < m * d; ++i) out[i] = (inverse ? W[i] * root : W[i] / root) + out[i];
}

// Dense T_A = sigma^-1/2 I + U diag(c) U^T (or T_A^-1 with inverse = 1), d x d.
void or_lowrank_T(const double *U, const double *mu, int64_t d, int64_t r, double sigma, int inverse, double *T) {
  std::vector<double> c(static_cast<size_t>(r)), Uc(static_cast<size_t>(d * r));
  lowrank_coeffs(mu, r, sigma, inverse, c.data());
  for (int64_t i = 0; i < d; ++i)
    for (int64_t j = 0; j < r; ++j) Uc[i * r + j] = U[i * r + j] * c[j];
  matmul_bt(Uc.data(), U, d, r, d, T);
  const double base = inverse ? std::sqrt(sigma) : 1.0 / std::sqrt(sigma);
  for (int64_t i = 0; i < d; ++i) T[i * d + i] += base;
}

// The completed factor U diag(mu - sigma) U^T + sigma I, d x d.
void or_lowrank_dense(const double *U, const double *mu, int64_t d, int64_t r, double sigma, double *A) {
  std::vector<double> Ul(static_cast<size_t>(d * r));
  for (int64_t i = 0; i < d; ++i)
    for (int64_t j = 0; j < r; ++j) Ul[i * r + j] = U[i * r + j] * (mu[j] - sigma);
  matmul_bt(Ul.data(), U, d, r, d, A);
  for (int64_t i = 0; i < d; ++i) A[i * d + i] += sigma;
}

// ---- error feedback (Algorithm 1: U~ = W~ + R; R <- U~ - Dequantize(Q(U~))) -----------

// out = fl32(a + b) element by element.
void or_add_f32(const float *a, const float *b, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = a[i] + b[i];
}

// out = fl32(a - b) element by element.
void or_sub_f32(const float *a, const float *b, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = a[i] - b[i];
}

// FP32 rounding (nearest even) of double values.
void or_round_f32(const double *x, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = static_cast<float>(x[i]);
}

// ---- fidelity ([notes] simplification 1, eq. (15): RelL2, Cos, MaxErr, MSE) -----------

// out[0..3] = RelL2, Cos, MaxErr, MSE of g_hat against g, in double.
void or_fidelity(const double *g_hat, const double *g, int64_t n, double *out) {
  double ee = 0.0, gg = 0.0, hh = 0.0, hg = 0.0, mx = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double e = g_hat[i] - g[i];
    ee += e * e;
    gg += g[i] * g[i];
    hh += g_hat[i] * g_hat[i];
    hg += g_hat[i] * g[i];
    if (std::fabs(e) > mx) mx = std::fabs(e);
  }
  const double nan = std::numeric_limits<double>::quiet_NaN();
  const double ng = std::sqrt(gg), nh = std::sqrt(hh);
  out[0] = ng > 0 ? std::sqrt(ee) / ng : nan;
  out[1] = (nh > 0 && ng > 0) ? hg / (nh * ng) : nan;
  out[2] = n ? mx : 0.0;
  out[3] = n ? ee / static_cast<double>(n) : 0.0;
}

// ---- the toy quantiser of the worked example ([notes] 玩具例子) ---------------------------

// Each coordinate to the nearest multiple of s / 8, s = max |v| (half to even).
void or_toy_quantize(const double *v, int64_t n, double *out) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i)
    if (std::fabs(v[i]) > s) s = std::fabs(v[i]);
  const double step = s / 8.0;
  for (int64_t i = 0; i < n; ++i) out[i] = std::nearbyint(v[i] / step) * step;
}

// Number of threads the build runs its parallel loops on (1 without OpenMP).
int or_threads(void) {
#ifdef _OPENMP
  int t = 1;
#pragma omp parallel
  {
#pragma omp single
    t = omp_get_num_threads();
  }
  return t;
#else
  return 1;
#endif
}

}  // extern "C"
