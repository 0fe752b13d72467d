"""CPU oracle for the GIFT per-layer gradient codec.  TEST INFRASTRUCTURE ONLY.

This file is the plain, slow and obviously correct statement of what the codec
computes.  It is used by the tests, by the smoke check and by the benchmark's
CPU-baseline leg; the product path (the CUDA library and its binding) never
imports it, and it imports nothing from the product.  It shares no code with
the CUDA kernels: the only thing both sides share is the seeded input generator
(fac_whitening_gb300/synth.py), which holds none of the method's arithmetic.

Sources, cited by page title and section (the pages give equations and an
algorithm, no code):
  [notes]    "GIFT 阅读笔记:量化用的坐标系,比量化器本身更重要" (GIFT reading notes,
             zhongzhuzhou.org, 2026-07-16).  Sections: 前置知识 (prerequisites, with
             "What FP8 is" and "K-FAC and the Fisher"), 核心想法 (core idea, steps 1-3,
             eqs. (5)-(14)), 三次简化 (three simplifications, eqs. (15)-(17) and the
             profiling procedure), 算法 1 (Algorithm 1), 玩具例子 (the worked 2x2 example,
             eqs. (A1)-(A3)).
  [abstract] "GIFT: Geometry-Informed Low-precision Gradient Communication for LLM
             Pretraining" (shd-paper.top summary), English abstract: names FP8 and
             NVFP4 as the low-precision formats.

Precision: every linear-algebra step runs in float64.  The quantiser is a
bit-exact contract, so its scalar steps are FP32 operations written one by one
(numpy float32 arithmetic is IEEE round-to-nearest-even, no fused multiply-add).

Readings taken where the pages are silent (each is listed in the design notes):
  * rounding to FP8/FP4 is round-to-nearest-even with saturation to the largest
    finite value ("satfinite"); the sign of zero is kept;
  * s = amax / FMAX is stored and elements are scaled by m = FMAX / amax, both
    single FP32 divisions; amax = 0 gives s = 0 and m = 0; an m that overflows
    FP32 is clamped to the largest finite FP32;
  * a non-finite element raises NonFinite;
  * the rank-r factor is completed with sigma * I, sigma the mean of the
    eigenvalues of A outside the top r (so that trace is preserved);
  * NVFP4 = E2M1 codes with one E4M3 scale per 16 consecutive elements of a row
    and one FP32 tensor scale (the pages name NVFP4 but give no layout);
  * replica reduce dequantises each replica with its own scale and averages in
    fixed replica order.

Functions whose results are not pinned to something outside this file are
marked "parity unpinned" in their docstring.  At present every function has a
pin in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F32_MAX = np.float32(np.finfo(np.float32).max)


class NonFinite(ValueError):
    """The input tensor holds a NaN or an infinity."""


class NotPositiveDefinite(ValueError):
    """A factor is not positive definite (Cholesky pivot or sigma <= 0)."""


# ======================================================================================
# Number formats  ([notes] 前置知识, "What FP8 is": E4M3 max about 448, E5M2 max about
# 57344, 2^3 or 2^2 mantissa levels per octave; [abstract] NVFP4)
# ======================================================================================

class Fmt:
    """A sign / exponent / mantissa minifloat with no infinities in its finite range."""

    def __init__(self, name, ebits, mbits, bias, maxval, nan_codes):
        self.name = name
        self.ebits = ebits
        self.mbits = mbits
        self.bias = bias
        self.maxval = float(maxval)
        self.emin = 1 - bias              # exponent of the smallest normal binade
        self.nbits = 1 + ebits + mbits
        self.nan_codes = nan_codes        # magnitude codes that decode to NaN/Inf

    @property
    def max_code(self) -> int:
        """Magnitude bits of the largest finite value."""
        return encode_scalar(self.maxval, self)

    @property
    def min_subnormal(self) -> float:
        return 2.0 ** (self.emin - self.mbits)


E4M3 = Fmt("e4m3", 4, 3, 7, 448.0, nan_codes=(0x7F,))
E5M2 = Fmt("e5m2", 5, 2, 15, 57344.0, nan_codes=(0x7C, 0x7D, 0x7E, 0x7F))
E2M1 = Fmt("e2m1", 2, 1, 1, 6.0, nan_codes=())

FORMATS = {"e4m3": E4M3, "e5m2": E5M2}


def round_to_format(y, fmt: Fmt) -> np.ndarray:
    """Round FP32 values to the nearest value of `fmt` (ties to even), saturating.

    Works on the exact values: each FP32 input is widened to float64, the
    quantum of its binade (or of the subnormal range) is a power of two, and
    np.rint rounds the quotient half-to-even.  Magnitudes at or above the
    largest finite value saturate to it.  NaN stays NaN.
    """
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, fmt.emin)          # binade exponent, clamped to the subnormal range
    q = np.ldexp(1.0, e - fmt.mbits)          # spacing of representable values there
    v = np.rint(a / q) * q
    v = np.where(a >= fmt.maxval, fmt.maxval, np.minimum(v, fmt.maxval))
    v = np.where(np.isnan(y), np.nan, v)
    return np.copysign(v, y)


def value_to_code(v, fmt: Fmt) -> np.ndarray:
    """Bit pattern of exactly representable values `v` (float64) of `fmt`."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.int64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= 2.0 ** fmt.emin
    e_field = np.where(normal, e + fmt.bias, 0)
    mant = np.where(normal,
                    a / np.ldexp(1.0, np.where(normal, e, 0) - fmt.mbits) - 2 ** fmt.mbits,
                    a / fmt.min_subnormal)
    mant = np.where(a == 0, 0, mant)
    e_field = np.where(a == 0, 0, e_field)
    code = (sign << (fmt.nbits - 1)) | (e_field.astype(np.int64) << fmt.mbits) | mant.astype(np.int64)
    nan_code = (1 << (fmt.nbits - 1)) - 1 if fmt.nan_codes else 0
    code = np.where(np.isnan(v), nan_code, code)
    return code.astype(np.uint8)


def encode(y, fmt: Fmt) -> np.ndarray:
    """FP32 -> code bytes of `fmt` (round to nearest even, satfinite)."""
    return value_to_code(round_to_format(y, fmt), fmt)


def encode_scalar(y: float, fmt: Fmt) -> int:
    return int(encode(np.array([y], dtype=np.float32), fmt)[0])


def decode(code, fmt: Fmt) -> np.ndarray:
    """Code bytes -> exact values (float64) from the sign / exponent / mantissa fields."""
    c = np.asarray(code, dtype=np.int64) & ((1 << fmt.nbits) - 1)
    sign = np.where((c >> (fmt.nbits - 1)) & 1, -1.0, 1.0)
    e_field = (c >> fmt.mbits) & ((1 << fmt.ebits) - 1)
    mant = c & ((1 << fmt.mbits) - 1)
    sub = mant * fmt.min_subnormal
    nor = (1.0 + mant / 2.0 ** fmt.mbits) * np.ldexp(1.0, e_field - fmt.bias)
    v = sign * np.where(e_field == 0, sub, nor)
    mag = c & ((1 << (fmt.nbits - 1)) - 1)
    if fmt.nan_codes:
        v = np.where(np.isin(mag, fmt.nan_codes), np.nan, v)
    if fmt.name == "e5m2":
        v = np.where(mag == 0x7C, sign * np.inf, v)
    return v


# ======================================================================================
# Scaling and FP8 quantisation  ([notes] 前置知识 "What FP8 is": s = amax(X)/FP8_MAX,
# per tensor or per block; Algorithm 1: Scale, Q, Dequantize)
# ======================================================================================

def abs_max(x) -> np.float32:
    """amax = max |x| (exact); raises NonFinite on NaN/Inf."""
    x = np.asarray(x, dtype=np.float32)
    if x.size == 0:
        return F32(0.0)
    if not np.all(np.isfinite(x)):
        raise NonFinite("non-finite element")
    return F32(np.max(np.abs(x)))


def scale_pair(amax, fmt: Fmt):
    """(s, m): s = amax / FMAX (stored scale) and m = FMAX / amax (multiplier).

    Each is one correctly rounded FP32 division.  amax = 0 gives (0, 0); an m
    beyond the FP32 range is clamped to the largest finite FP32.
    """
    amax = F32(amax)
    fmax = F32(fmt.maxval)
    if amax == 0:
        return F32(0.0), F32(0.0)
    with np.errstate(over="ignore"):
        s = F32(amax / fmax)
        m = F32(fmax / amax)
    if np.isinf(m):
        m = F32_MAX
    return s, m


def quantize_with_multiplier(x, m, fmt: Fmt) -> np.ndarray:
    """code = RNE_satfinite(fl32(x * m))."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        y = (x * F32(m)).astype(np.float32)
    return encode(y, fmt)


def dequantize(codes, s, fmt: Fmt) -> np.ndarray:
    """x_hat = fl32(value(code) * s)."""
    v = decode(codes, fmt).astype(np.float32)
    return (v * np.asarray(s, dtype=np.float32)).astype(np.float32)


def quantize_tensor(x, fmt: Fmt, amax=None):
    """Per-tensor scaling: returns (codes uint8 same shape, s float32, amax used).

    `amax` overrides the tensor's own amax (the AllReduceMax'd shared scale of
    the Euclidean path in Algorithm 1).
    """
    x = np.asarray(x, dtype=np.float32)
    local = abs_max(x)
    a = local if amax is None else F32(amax)
    s, m = scale_pair(a, fmt)
    return quantize_with_multiplier(x, m, fmt), s, a


BLOCK = 128


def block_grid(d_out, d_in, b=BLOCK):
    return (d_out + b - 1) // b, (d_in + b - 1) // b


def block_amax(x, b=BLOCK) -> np.ndarray:
    """amax of every b x b tile (edge tiles clipped), shape (ceil(d_out/b), ceil(d_in/b))."""
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise NonFinite("non-finite element")
    nbr, nbc = block_grid(*x.shape, b)
    out = np.zeros((nbr, nbc), dtype=np.float32)
    for i in range(nbr):
        for j in range(nbc):
            t = x[i * b:(i + 1) * b, j * b:(j + 1) * b]
            out[i, j] = np.max(np.abs(t)) if t.size else 0.0
    return out


def quantize_block128(x, fmt: Fmt, amax=None):
    """Per-block scaling on 128 x 128 tiles: returns (codes, scales[nbr, nbc], amax[nbr, nbc])."""
    x = np.asarray(x, dtype=np.float32)
    am = block_amax(x) if amax is None else np.asarray(amax, dtype=np.float32)
    nbr, nbc = am.shape
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros((nbr, nbc), dtype=np.float32)
    for i in range(nbr):
        for j in range(nbc):
            s, m = scale_pair(am[i, j], fmt)
            scales[i, j] = s
            sl = (slice(i * BLOCK, (i + 1) * BLOCK), slice(j * BLOCK, (j + 1) * BLOCK))
            codes[sl] = quantize_with_multiplier(x[sl], m, fmt)
    return codes, scales, am


def dequantize_block128(codes, scales, fmt: Fmt) -> np.ndarray:
    codes = np.asarray(codes)
    out = np.zeros(codes.shape, dtype=np.float32)
    nbr, nbc = scales.shape
    for i in range(nbr):
        for j in range(nbc):
            sl = (slice(i * BLOCK, (i + 1) * BLOCK), slice(j * BLOCK, (j + 1) * BLOCK))
            out[sl] = dequantize(codes[sl], scales[i, j], fmt)
    return out


# 1-D blocks: the per-block Euclidean baseline of the experiments (block size 512).  Reading:
# one FP32 scale per 512 consecutive elements of the row-major flattened tensor, the last
# block shorter when the element count is not a multiple of 512.
BLOCK1D = 512


def quantize_block1d(x, fmt: Fmt, amax=None, b=BLOCK1D):
    """Returns (codes, scales[nb], amax[nb]), nb = ceil(n / b); amax overrides the blocks'
    own (one value per block)."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.ravel()
    nb = (flat.size + b - 1) // b
    codes = np.zeros(flat.size, dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    am = np.zeros(nb, dtype=np.float32)
    for i in range(nb):
        blk = flat[i * b:(i + 1) * b]
        am[i] = abs_max(blk) if amax is None else F32(np.asarray(amax).ravel()[i])
        s, m = scale_pair(am[i], fmt)
        scales[i] = s
        codes[i * b:(i + 1) * b] = quantize_with_multiplier(blk, m, fmt)
    return codes.reshape(x.shape), scales, am


def dequantize_block1d(codes, scales, fmt: Fmt, b=BLOCK1D) -> np.ndarray:
    codes = np.asarray(codes)
    flat = codes.ravel()
    out = np.zeros(flat.size, dtype=np.float32)
    for i in range(len(scales)):
        out[i * b:(i + 1) * b] = dequantize(flat[i * b:(i + 1) * b], scales[i], fmt)
    return out.reshape(codes.shape)


# ======================================================================================
# NVFP4 ([abstract]: "FP8 and NVFP4"; the layout below is the plain public reading:
# E2M1 codes, one E4M3 scale per 16 consecutive elements of a row, one FP32 tensor scale)
# ======================================================================================

NV_GROUP = 16
NV_TENSOR_DIV = F32(448.0 * 6.0)    # 2688, exact in FP32


def quantize_nvfp4(x, amax=None):
    """Returns (codes uint8 [d_out, d_in/2] packed, block scales uint8 [d_out, d_in/16],
    tensor scale float32, tensor amax used).

    s_t = amax / 2688.  For each group of 16 consecutive elements of a row with
    group amax a_b: e_b = E4M3(a_b / fl32(6 s_t)), eff = fl32(e_b * s_t),
    r_b = 1 / eff (eff = 0 gives r_b = 0; an r_b beyond FP32 is clamped), and the
    element code is E2M1(fl32(x * r_b)).  The even column goes to the low nibble.
    """
    x = np.asarray(x, dtype=np.float32)
    d_out, d_in = x.shape
    if d_in % NV_GROUP:
        raise ValueError("NVFP4 needs d_in to be a multiple of 16")
    local = abs_max(x)
    at = local if amax is None else F32(amax)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        s_t = F32(at / NV_TENSOR_DIV)
        g = x.reshape(d_out, d_in // NV_GROUP, NV_GROUP)
        ab = np.max(np.abs(g), axis=2).astype(np.float32)
        six_st = F32(F32(6.0) * s_t)
        if s_t == 0:
            ratio = np.zeros_like(ab)
        else:
            ratio = (ab / six_st).astype(np.float32)
        eb_codes = encode(ratio, E4M3)
        eb = decode(eb_codes, E4M3).astype(np.float32)
        eff = (eb * s_t).astype(np.float32)
        rb = np.where(eff == 0, F32(0.0), (F32(1.0) / np.where(eff == 0, F32(1.0), eff))).astype(np.float32)
        rb = np.where(np.isinf(rb), F32_MAX, rb).astype(np.float32)
        y = (g * rb[:, :, None]).astype(np.float32)
    c = encode(y, E2M1).reshape(d_out, d_in).astype(np.uint8)
    packed = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), eb_codes.astype(np.uint8), s_t, at


def dequantize_nvfp4(packed, block_scales, s_t) -> np.ndarray:
    """x_hat = fl32(fl32(value(code) * value(e_b)) * s_t)."""
    packed = np.asarray(packed, dtype=np.uint8)
    d_out = packed.shape[0]
    d_in = packed.shape[1] * 2
    c = np.zeros((d_out, d_in), dtype=np.uint8)
    c[:, 0::2] = packed & 0xF
    c[:, 1::2] = packed >> 4
    v = decode(c, E2M1).astype(np.float32).reshape(d_out, d_in // NV_GROUP, NV_GROUP)
    eb = decode(block_scales, E4M3).astype(np.float32)
    p = (v * eb[:, :, None]).astype(np.float32)
    return (p * F32(s_t)).astype(np.float32).reshape(d_out, d_in)


# ======================================================================================
# Generic quantise / dequantise front end (format x scaling)
# ======================================================================================

def quantize(x, fmt: str, scaling: str = "tensor", amax=None):
    """Returns a dict with 'codes', 'scales' (FP32 per tensor/block, or E4M3 bytes for
    NVFP4), 'tensor_scale' (NVFP4 only) and 'amax'."""
    if fmt == "f32":
        return {"codes": np.asarray(x, dtype=np.float32).copy(), "scales": None,
                "tensor_scale": None, "amax": None}
    if fmt == "nvfp4":
        c, bs, st, at = quantize_nvfp4(x, amax)
        return {"codes": c, "scales": bs, "tensor_scale": st, "amax": at}
    f = FORMATS[fmt]
    if scaling == "tensor":
        c, s, a = quantize_tensor(x, f, amax)
        return {"codes": c, "scales": np.array([s], dtype=np.float32), "tensor_scale": None, "amax": a}
    if scaling == "block512":
        c, s, a = quantize_block1d(x, f, amax)
        return {"codes": c, "scales": s, "tensor_scale": None, "amax": a}
    c, s, a = quantize_block128(x, f, amax)
    return {"codes": c, "scales": s, "tensor_scale": None, "amax": a}


def dequantize_any(q, fmt: str, scaling: str = "tensor") -> np.ndarray:
    if fmt == "f32":
        return np.asarray(q["codes"], dtype=np.float32)
    if fmt == "nvfp4":
        return dequantize_nvfp4(q["codes"], q["scales"], q["tensor_scale"])
    f = FORMATS[fmt]
    if scaling == "tensor":
        return dequantize(q["codes"], q["scales"][0], f)
    if scaling == "block512":
        return dequantize_block1d(q["codes"], q["scales"], f)
    return dequantize_block128(q["codes"], q["scales"], f)


# ======================================================================================
# Replica reduce: the data-parallel average of eq. (1) ([notes] 前置知识, data parallel),
# taken over dequantised replicas as in Algorithm 1 (AllReduceSum, Dequantize, / N)
# ======================================================================================

def replica_reduce(qs, fmt: str, scaling: str = "tensor") -> np.ndarray:
    """out = (deq_0 + deq_1 + ... + deq_{R-1}) / R, FP32 additions left to right."""
    R = len(qs)
    acc = None
    for q in qs:
        d = dequantize_any(q, fmt, scaling)
        # acc starts at replica 0's values (not at 0 + deq_0, which would turn -0 into +0)
        acc = d.copy() if acc is None else (acc + d).astype(np.float32)
    return (acc / F32(R)).astype(np.float32)


# ======================================================================================
# Boundary-hit profiler ([notes] 三次简化, simplification 3: encode the flattened gradient
# with the scale that would be used and count values hitting the upper or lower
# boundary of the FP8 format; the sum of the two rates is the fragility score)
# ======================================================================================

def boundary_hits(x, fmt: str, scaling: str = "tensor"):
    """Returns (upper, lower, n): upper = #{|code| == largest finite code},
    lower = #{x != 0 and |code| == 0}, n = number of elements."""
    x = np.asarray(x, dtype=np.float32)
    f = FORMATS[fmt]
    q = quantize(x, fmt, scaling)
    mag = q["codes"].astype(np.int64) & 0x7F
    upper = int(np.count_nonzero(mag == f.max_code))
    lower = int(np.count_nonzero((x != 0) & (mag == 0)))
    return upper, lower, int(x.size)


def fragility_score(hits) -> float:
    upper, lower, n = hits
    return (upper + lower) / n if n else 0.0


def select_fragile(scores, k):
    """Indices of the k highest scores; ties go to the lower layer index."""
    order = sorted(range(len(scores)), key=lambda i: (-scores[i], i))
    return order[:k]


def window_scores(counts):
    """Fragility score of every layer over a profiling window (the profiling procedure of
    simplification 3: boundary-hit rates averaged over the window, upper and lower summed).
    counts[l] = (upper, lower, n) summed over the window's steps.  A layer's element count
    is the same at every step, so the window mean of the per-step rate (upper + lower) / n
    is the summed hits over the summed n."""
    return [fragility_score(c) for c in counts]


def knee_count(ranked, k_min=1, k_max=None):
    """The number of layers before the clear drop in score (simplification 3, Figure 3: the
    fragile group, then a marked drop).  Reading: over k in [k_min, min(k_max, L - 1)],
    the k with the largest drop ranked[k-1] - ranked[k] between consecutive scores in
    descending order; equal drops go to the smaller k.  With one layer, or k_min = L, the
    answer is L."""
    L = len(ranked)
    k_max = L if k_max is None else k_max
    if not 1 <= k_min <= k_max <= L:
        raise ValueError("need 1 <= k_min <= k_max <= number of layers")
    if k_min == L:
        return L
    best_k, best = k_min, None
    for k in range(k_min, min(k_max, L - 1) + 1):
        drop = ranked[k - 1] - ranked[k]
        if best is None or drop > best:
            best_k, best = k, drop
    return best_k


def select_fragile_knee(scores, k_min=1, k_max=None):
    """Layer indices by descending score (ties to the lower index), cut at the knee."""
    order = sorted(range(len(scores)), key=lambda i: (-scores[i], i))
    k = knee_count([scores[i] for i in order], k_min, k_max)
    return order[:k]


# ======================================================================================
# K-FAC factors ([notes] 前置知识 "K-FAC", eq. (4): A = E[a a^T], G = E[delta delta^T])
# ======================================================================================

def kfac_factor(a) -> np.ndarray:
    """A = a^T a / T in float64 (inputs widened exactly)."""
    a = np.asarray(a, dtype=np.float64)
    return (a.T @ a) / a.shape[0]


def cholesky(A) -> np.ndarray:
    """Textbook Cholesky A = L L^T ([notes] 核心想法 step 2, eq. (7)), column by column."""
    A = np.asarray(A, dtype=np.float64)
    n = A.shape[0]
    L = np.zeros_like(A)
    for j in range(n):
        d = A[j, j] - np.dot(L[j, :j], L[j, :j])
        if not d > 0:
            raise NotPositiveDefinite(f"pivot {j} = {d}")
        L[j, j] = np.sqrt(d)
        L[j + 1:, j] = (A[j + 1:, j] - L[j + 1:, :j] @ L[j, :j]) / L[j, j]
    return L


def lower_inverse(L) -> np.ndarray:
    """L^-1 of a lower-triangular L by forward substitution, column by column of I."""
    L = np.asarray(L, dtype=np.float64)
    n = L.shape[0]
    X = np.zeros_like(L)
    for i in range(n):
        # row i of L X = I:  L[i,i] X[i,:] = e_i - L[i,:i] X[:i,:]
        rhs = -(L[i, :i] @ X[:i, :])
        rhs[i] += 1.0
        X[i, :] = rhs / L[i, i]
    return X


def solve_right_lower_t(W, L) -> np.ndarray:
    """X with X L^T = W (i.e. X = W L^-T), forward substitution over the columns of X."""
    W = np.asarray(W, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    X = np.zeros_like(W)
    for j in range(L.shape[0]):
        X[:, j] = (W[:, j] - X[:, :j] @ L[j, :j]) / L[j, j]
    return X


def solve_left_lower(L, W) -> np.ndarray:
    """Y with L Y = W (i.e. Y = L^-1 W), forward substitution over the rows of Y."""
    W = np.asarray(W, dtype=np.float64)
    L = np.asarray(L, dtype=np.float64)
    Y = np.zeros_like(W)
    for i in range(L.shape[0]):
        Y[i, :] = (W[i, :] - L[i, :i] @ Y[:i, :]) / L[i, i]
    return Y


# ---- symmetric eigensolver ------------------------------------------------------------

def jacobi_eigh(S, tol=1e-15, max_sweeps=40):
    """Cyclic Jacobi eigendecomposition of a symmetric matrix (float64).

    Each rotation zeroes one off-diagonal pair (p, q) with the classical choice
    of the smaller rotation angle (Golub & Van Loan, "Matrix Computations",
    section 8.5).  Returns (eigenvalues descending, eigenvectors as columns).
    """
    A = np.array(S, dtype=np.float64, copy=True)
    n = A.shape[0]
    V = np.eye(n)
    for _ in range(max_sweeps):
        off = np.sqrt(np.sum(np.tril(A, -1) ** 2))
        scale = np.sqrt(np.sum(A * A))
        if off <= tol * max(scale, 1e-300):
            break
        for p in range(n - 1):
            for q in range(p + 1, n):
                apq = A[p, q]
                if abs(apq) <= 1e-18 * np.sqrt(abs(A[p, p] * A[q, q])) or apq == 0.0:
                    continue
                theta = (A[q, q] - A[p, p]) / (2.0 * apq)
                t = np.sign(theta) / (abs(theta) + np.sqrt(theta * theta + 1.0)) if theta != 0 else 1.0
                c = 1.0 / np.sqrt(t * t + 1.0)
                s = t * c
                # A <- J^T A J with J the rotation in the (p, q) plane
                ap = A[:, p].copy()
                aq = A[:, q].copy()
                A[:, p] = c * ap - s * aq
                A[:, q] = s * ap + c * aq
                ap = A[p, :].copy()
                aq = A[q, :].copy()
                A[p, :] = c * ap - s * aq
                A[q, :] = s * ap + c * aq
                A[p, q] = A[q, p] = 0.0
                vp = V[:, p].copy()
                vq = V[:, q].copy()
                V[:, p] = c * vp - s * vq
                V[:, q] = s * vp + c * vq
    w = np.diag(A).copy()
    order = np.argsort(-w, kind="stable")
    return w[order], V[:, order]


def subspace_iteration(apply_A, n, k=64, iters=16, seed=12345):
    """Top-k Ritz pairs of a symmetric PSD operator by block subspace iteration.

    Q0 = orth(Omega) with Omega iid N(0,1) n x k; Q_{i+1} = orth(A Q_i) (QR is the
    library Householder QR); finally B = Q^T A Q and its Jacobi eigenpairs give
    mu and U = Q V (N. Halko, P.-G. Martinsson, J. Tropp, "Finding structure with
    randomness", SIAM Review 2011, Alg. 4.4 plus Rayleigh-Ritz).
    """
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((n, k)))
    for _ in range(iters):
        Q, _ = np.linalg.qr(apply_A(Q))
    B = Q.T @ apply_A(Q)
    B = 0.5 * (B + B.T)
    mu, V = jacobi_eigh(B)
    return mu, Q @ V


class LowRankFactor:
    """A ~ U diag(lambda) U^T + sigma I with mu = lambda + sigma the top-r eigenvalues.

    ([notes] 三次简化 simplification 2, eq. (17): A ~ U_r Lambda_r U_r^T, r = 32.  The
    sigma I completion makes the input-side transform invertible; sigma is the
    mean of the remaining eigenvalues, tr(A) - sum(mu) over d_in - r, so the
    completed factor keeps tr(A).  With r = d_in, sigma cancels and is set to 1.)
    """

    def __init__(self, U, mu, sigma):
        self.U = np.asarray(U, dtype=np.float64)
        self.mu = np.asarray(mu, dtype=np.float64)
        self.sigma = float(sigma)

    @property
    def rank(self):
        return self.mu.shape[0]

    @property
    def lam(self):
        return self.mu - self.sigma

    def dense(self):
        d = self.U.shape[0]
        return (self.U * self.lam) @ self.U.T + self.sigma * np.eye(d)


def lowrank_from_eigs(mu_all, V_all, trace, d_in, r) -> LowRankFactor:
    mu = np.asarray(mu_all[:r], dtype=np.float64)
    U = np.asarray(V_all[:, :r], dtype=np.float64)
    if r == d_in:
        sigma = 1.0
    else:
        sigma = (trace - np.sum(mu)) / (d_in - r)
    if not (sigma > 0 and np.all(mu > 0)):
        raise NotPositiveDefinite(f"sigma = {sigma}, min mu = {np.min(mu)}")
    return LowRankFactor(U, mu, sigma)


def lowrank_factor_from_A(A, r=32, k=64, iters=16, seed=12345) -> LowRankFactor:
    """Rank-r factor of an explicit A: exact Jacobi when d_in <= 128, else subspace iteration."""
    A = np.asarray(A, dtype=np.float64)
    d = A.shape[0]
    tr = float(np.trace(A))
    if d <= 128:
        mu, V = jacobi_eigh(A)
    else:
        mu, V = subspace_iteration(lambda X: A @ X, d, k=min(k, d), iters=iters, seed=seed)
    return lowrank_from_eigs(mu, V, tr, d, r)


def lowrank_factor_from_activations(a, r=32, k=64, iters=16, seed=12345) -> LowRankFactor:
    """Rank-r factor of A = a^T a / T without forming A (A x = a^T (a x) / T)."""
    a64 = np.asarray(a, dtype=np.float64)
    T, d = a64.shape
    tr = float(np.sum(a64 * a64)) / T
    if d <= 128:
        return lowrank_factor_from_A(kfac_factor(a64), r=r)
    mu, V = subspace_iteration(lambda X: a64.T @ (a64 @ X) / T, d, k=min(k, d), iters=iters, seed=seed)
    return lowrank_from_eigs(mu, V, tr, d, r)


# ======================================================================================
# Transforms ([notes] 核心想法 step 3, eqs. (11)-(14); 三次简化 simplification 1, eq. (16):
# W~ = W_g T_A with T_A from the input-side factor; Algorithm 1 maps back with L_A^T)
# ======================================================================================

def lowrank_coeffs(F: LowRankFactor, inverse=False):
    """c_i = mu_i^-1/2 - sigma^-1/2 (whitening) or mu_i^1/2 - sigma^1/2 (map back)."""
    if inverse:
        return np.sqrt(F.mu) - np.sqrt(F.sigma)
    return 1.0 / np.sqrt(F.mu) - 1.0 / np.sqrt(F.sigma)


def lowrank_T(F: LowRankFactor, inverse=False) -> np.ndarray:
    """Dense T_A = sigma^-1/2 I + U (diag(mu^-1/2) - sigma^-1/2) U^T (or its inverse)."""
    d = F.U.shape[0]
    c = lowrank_coeffs(F, inverse)
    base = np.sqrt(F.sigma) if inverse else 1.0 / np.sqrt(F.sigma)
    return base * np.eye(d) + (F.U * c) @ F.U.T


def lowrank_whiten(W, F: LowRankFactor) -> np.ndarray:
    """W~ = W T_A = sigma^-1/2 W + ((W U) diag(c)) U^T."""
    W = np.asarray(W, dtype=np.float64)
    c = lowrank_coeffs(F)
    return W / np.sqrt(F.sigma) + ((W @ F.U) * c) @ F.U.T


def lowrank_unwhiten(X, F: LowRankFactor) -> np.ndarray:
    """W_hat = X T_A^-1 = sigma^1/2 X + ((X U) diag(c')) U^T."""
    X = np.asarray(X, dtype=np.float64)
    c = lowrank_coeffs(F, inverse=True)
    return X * np.sqrt(F.sigma) + ((X @ F.U) * c) @ F.U.T


def chol_input_whiten(W, LA) -> np.ndarray:
    """W~ = W L_A^-T (input side only, eq. (16) with T_A = L_A^-T)."""
    return solve_right_lower_t(W, LA)


def chol_two_sided_whiten(W, LG, LA) -> np.ndarray:
    """W~ = L_G^-1 W L_A^-T (eq. (11))."""
    return solve_right_lower_t(solve_left_lower(LG, W), LA)


def chol_input_unwhiten(X, LA) -> np.ndarray:
    """W_hat = X L_A^T."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(LA, dtype=np.float64).T


def chol_two_sided_unwhiten(X, LG, LA) -> np.ndarray:
    """W_hat = L_G X L_A^T (eq. (14))."""
    return np.asarray(LG, dtype=np.float64) @ np.asarray(X, dtype=np.float64) @ np.asarray(LA, dtype=np.float64).T


def chol_whiten_with_inverses(W, LAinv, LGinv=None) -> np.ndarray:
    """W~ = L_G^-1 W L_A^-T written with given inverse factors (eq. (11) as printed, with
    L^-1; the input-side form of eq. (16) when LGinv is None)."""
    X = np.asarray(W, dtype=np.float64) @ np.asarray(LAinv, dtype=np.float64).T
    if LGinv is not None:
        X = np.asarray(LGinv, dtype=np.float64) @ X
    return X


class Xform:
    """A transform: kind in {identity, lowrank, chol_input, chol_two_sided} and its factor.

    For the Cholesky kinds the factor may carry the inverse factors L^-1 explicitly
    (as libgift's factor does); the whitening then multiplies by them, otherwise it
    solves with L.
    """

    def __init__(self, kind, F=None, LA=None, LG=None, LAinv=None, LGinv=None):
        self.kind, self.F, self.LA, self.LG = kind, F, LA, LG
        self.LAinv, self.LGinv = LAinv, LGinv

    def whiten(self, W):
        if self.kind == "identity":
            return np.asarray(W, dtype=np.float64)
        if self.kind == "lowrank":
            return lowrank_whiten(W, self.F)
        if self.kind == "chol_input":
            if self.LAinv is not None:
                return chol_whiten_with_inverses(W, self.LAinv)
            return chol_input_whiten(W, self.LA)
        if self.LAinv is not None and self.LGinv is not None:
            return chol_whiten_with_inverses(W, self.LAinv, self.LGinv)
        return chol_two_sided_whiten(W, self.LG, self.LA)

    def unwhiten(self, X):
        if self.kind == "identity":
            return np.asarray(X, dtype=np.float64)
        if self.kind == "lowrank":
            return lowrank_unwhiten(X, self.F)
        if self.kind == "chol_input":
            return chol_input_unwhiten(X, self.LA)
        return chol_two_sided_unwhiten(X, self.LG, self.LA)


# ======================================================================================
# The codec end to end (Algorithm 1, geometry-aware branch and Euclidean path)
# ======================================================================================

def encode_layer(W, xf: Xform, fmt: str, scaling="tensor", amax=None, residual=None):
    """Whiten, optionally add the error-feedback residual, scale and quantise.

    Returns (q, transformed FP32, new residual or None).  The transformed tensor
    is rounded to FP32 before quantisation.  With a residual buffer R:
    U~ = W~ + R, quantise U~, R <- U~ - Dequantize(Q(U~)) (Algorithm 1, error
    feedback in the whitened coordinates).
    """
    Wt = xf.whiten(W).astype(np.float32)
    if residual is not None:
        Wt = (Wt + np.asarray(residual, dtype=np.float32)).astype(np.float32)
    q = quantize(Wt, fmt, scaling, amax)
    new_res = None
    if residual is not None:
        new_res = (Wt - dequantize_any(q, fmt, scaling)).astype(np.float32)
    return q, Wt, new_res


def decode_layer(X, xf: Xform) -> np.ndarray:
    """Map the reduced (or dequantised) whitened tensor back: W_hat = X T_A^-1."""
    return xf.unwhiten(X)


# ======================================================================================
# Fidelity ([notes] 三次简化 simplification 1, eq. (15): RelL2, Cos, MaxErr, MSE)
# ======================================================================================

def fidelity(g_hat, g):
    g_hat = np.asarray(g_hat, dtype=np.float64).ravel()
    g = np.asarray(g, dtype=np.float64).ravel()
    e = g_hat - g
    ng = np.linalg.norm(g)
    nh = np.linalg.norm(g_hat)
    return {
        "rel_l2": float(np.linalg.norm(e) / ng) if ng > 0 else float("nan"),
        "cos": float(np.dot(g_hat, g) / (nh * ng)) if nh > 0 and ng > 0 else float("nan"),
        "max_err": float(np.max(np.abs(e))) if e.size else 0.0,
        "mse": float(np.dot(e, e) / e.size) if e.size else 0.0,
    }


# ======================================================================================
# The toy quantiser of the worked example ([notes] 玩具例子, step 4): round each
# coordinate to the nearest multiple of s/8 with s = max |.| of the vector
# ======================================================================================

def toy_quantize(v):
    v = np.asarray(v, dtype=np.float64)
    s = np.max(np.abs(v))
    step = s / 8.0
    return np.round(v / step) * step
