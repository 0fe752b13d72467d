"""The C++ statement of the oracle (gift_oracle.cpp), with the same Python API as the numpy
statement in gift_oracle.py.  TEST INFRASTRUCTURE ONLY.

Every step of the arithmetic runs in the C++ library; this module only converts arrays
(to contiguous float32 / float64 / uint8 buffers, exact widenings) and dispatches.  The
single-threaded build is the default; `use_openmp(True)` switches to the OpenMP build of the
same source, whose results are identical.  The library is built by oracle/build_oracle.py
(called by the package build) and loaded on first use.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build_oracle

F32 = np.float32
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_i32p = ctypes.POINTER(ctypes.c_int)
_i64 = ctypes.c_int64
APPLY_FN = ctypes.CFUNCTYPE(None, _f64p, _i64, _i64, _f64p, ctypes.c_void_p)

_LIBS = {}
_OPENMP = False


class NonFinite(ValueError):
    """The input tensor holds a NaN or an infinity."""


class NotPositiveDefinite(ValueError):
    """A factor is not positive definite (Cholesky pivot or sigma <= 0)."""


def _declare(lib):
    sig = {
        "or_format_info": (None, [ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _f64p]),
        "or_encode": (None, [_f32p, _i64, ctypes.c_int, _u8p]),
        "or_decode": (None, [_u8p, _i64, ctypes.c_int, _f64p]),
        "or_abs_max": (ctypes.c_int, [_f32p, _i64, _f32p]),
        "or_scale_pair": (None, [ctypes.c_float, ctypes.c_int, _f32p, _f32p]),
        "or_quantize_with_multiplier": (None, [_f32p, _i64, ctypes.c_float, ctypes.c_int, _u8p]),
        "or_dequantize": (None, [_u8p, _i64, ctypes.c_float, ctypes.c_int, _f32p]),
        "or_quantize_tensor": (ctypes.c_int, [_f32p, _i64, ctypes.c_int, _f32p, _u8p, _f32p, _f32p]),
        "or_block_amax": (ctypes.c_int, [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p]),
        "or_quantize_block2d": (ctypes.c_int, [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p,
                                                _u8p, _f32p, _f32p]),
        "or_dequantize_block2d": (None, [_u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int, _f32p]),
        "or_quantize_block1d": (ctypes.c_int, [_f32p, _i64, ctypes.c_int, ctypes.c_int, _f32p, _u8p, _f32p, _f32p]),
        "or_dequantize_block1d": (None, [_u8p, _i64, ctypes.c_int, _f32p, ctypes.c_int, _f32p]),
        "or_quantize_nvfp4": (ctypes.c_int, [_f32p, ctypes.c_int, ctypes.c_int, _f32p, _u8p, _u8p, _f32p, _f32p]),
        "or_dequantize_nvfp4": (None, [_u8p, _u8p, ctypes.c_float, ctypes.c_int, ctypes.c_int, _f32p]),
        "or_replica_mean": (None, [_f32p, ctypes.c_int, _i64, _f32p]),
        "or_boundary_counts": (None, [_f32p, _u8p, _i64, ctypes.c_int, _u64p]),
        "or_window_scores": (None, [_u64p, ctypes.c_int, _f64p]),
        "or_rank_layers": (None, [_f64p, ctypes.c_int, _i32p]),
        "or_knee_count": (ctypes.c_int, [_f64p, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
        "or_kfac_factor": (None, [_f64p, _i64, _i64, _f64p]),
        "or_trace": (ctypes.c_double, [_f64p, _i64]),
        "or_activation_trace": (ctypes.c_double, [_f64p, _i64, _i64]),
        "or_cholesky": (ctypes.c_int, [_f64p, _i64, _f64p]),
        "or_lower_inverse": (None, [_f64p, _i64, _f64p]),
        "or_solve_right_lower_t": (None, [_f64p, _f64p, _i64, _i64, _f64p]),
        "or_solve_left_lower": (None, [_f64p, _f64p, _i64, _i64, _f64p]),
        "or_matmul": (None, [_f64p, _f64p, _i64, _i64, _i64, _f64p]),
        "or_matmul_bt": (None, [_f64p, _f64p, _i64, _i64, _i64, _f64p]),
        "or_jacobi_eigh": (ctypes.c_int, [_f64p, _i64, ctypes.c_double, ctypes.c_int, _f64p, _f64p]),
        "or_subspace_iteration": (None, [ctypes.c_int, _f64p, _i64, _i64, _i64, ctypes.c_int, _f64p, APPLY_FN,
                                         ctypes.c_void_p, _f64p, _f64p]),
        "or_lowrank_from_eigs": (ctypes.c_int, [_f64p, _f64p, _i64, ctypes.c_double, _i64, _i64, _f64p, _f64p,
                                                _f64p]),
        "or_lowrank_apply": (None, [_f64p, _i64, _i64, _f64p, _f64p, _i64, ctypes.c_double, ctypes.c_int, _f64p]),
        "or_lowrank_T": (None, [_f64p, _f64p, _i64, _i64, ctypes.c_double, ctypes.c_int, _f64p]),
        "or_lowrank_dense": (None, [_f64p, _f64p, _i64, _i64, ctypes.c_double, _f64p]),
        "or_add_f32": (None, [_f32p, _f32p, _i64, _f32p]),
        "or_sub_f32": (None, [_f32p, _f32p, _i64, _f32p]),
        "or_round_f32": (None, [_f64p, _i64, _f32p]),
        "or_fidelity": (None, [_f64p, _f64p, _i64, _f64p]),
        "or_toy_quantize": (None, [_f64p, _i64, _f64p]),
        "or_threads": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def lib():
    """The loaded library (single-threaded, or the OpenMP build after use_openmp(True))."""
    key = "omp" if _OPENMP else "serial"
    if key not in _LIBS:
        path = build_oracle.LIB_OMP if _OPENMP else build_oracle.LIB_SERIAL
        if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(build_oracle.SRC):
            build_oracle.build(openmp=_OPENMP)
        _LIBS[key] = _declare(ctypes.CDLL(path))
    return _LIBS[key]


def use_openmp(on: bool) -> int:
    """Select the OpenMP build (True) or the single-threaded one; returns its thread count."""
    global _OPENMP
    _OPENMP = bool(on)
    return int(lib().or_threads())


# ---- marshalling helpers ---------------------------------------------------------------

def _c32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _c64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _cu8(x):
    return np.ascontiguousarray(x, dtype=np.uint8)


def _p(a, t):
    return a.ctypes.data_as(t)


def _opt32(x, n=None):
    if x is None:
        return None, None
    a = _c32(np.atleast_1d(np.asarray(x, dtype=np.float32)).ravel())
    return a, _p(a, _f32p)


# ---- number formats ----------------------------------------------------------------------

class Fmt:
    """Descriptor of a format of the C++ library (0 = E4M3, 1 = E5M2, 2 = E2M1); its
    constants are read from the library."""

    def __init__(self, name, fid):
        self.name, self.fid = name, fid
        e, m, b, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        mx = ctypes.c_double()
        lib().or_format_info(fid, ctypes.byref(e), ctypes.byref(m), ctypes.byref(b), ctypes.byref(n),
                             ctypes.byref(mx))
        self.ebits, self.mbits, self.bias, self.nbits, self.maxval = e.value, m.value, b.value, n.value, mx.value
        self.emin = 1 - self.bias

    @property
    def max_code(self) -> int:
        return int(encode(np.array([self.maxval], dtype=np.float32), self)[0])

    @property
    def min_subnormal(self) -> float:
        return 2.0 ** (self.emin - self.mbits)


class _Formats(dict):
    def __missing__(self, key):
        raise KeyError(key)


E4M3 = None
E5M2 = None
E2M1 = None
FORMATS = _Formats()


def _init_formats():
    global E4M3, E5M2, E2M1
    E4M3, E5M2, E2M1 = Fmt("e4m3", 0), Fmt("e5m2", 1), Fmt("e2m1", 2)
    FORMATS.update({"e4m3": E4M3, "e5m2": E5M2})


def encode(y, fmt: Fmt) -> np.ndarray:
    y = _c32(y)
    out = np.empty(y.shape, dtype=np.uint8)
    lib().or_encode(_p(y, _f32p), y.size, fmt.fid, _p(out, _u8p))
    return out


def encode_scalar(y: float, fmt: Fmt) -> int:
    return int(encode(np.array([y], dtype=np.float32), fmt)[0])


def decode(code, fmt: Fmt) -> np.ndarray:
    c = _cu8(np.asarray(code).astype(np.int64) & 0xFF)
    out = np.empty(c.shape, dtype=np.float64)
    lib().or_decode(_p(c, _u8p), c.size, fmt.fid, _p(out, _f64p))
    return out


# ---- scaling and quantisation -------------------------------------------------------------

def abs_max(x) -> np.float32:
    x = _c32(x)
    out = ctypes.c_float()
    if lib().or_abs_max(_p(x, _f32p), x.size, ctypes.byref(out)):
        raise NonFinite("non-finite element")
    return F32(out.value)


def scale_pair(amax, fmt: Fmt):
    s, m = ctypes.c_float(), ctypes.c_float()
    lib().or_scale_pair(float(F32(amax)), fmt.fid, ctypes.byref(s), ctypes.byref(m))
    return F32(s.value), F32(m.value)


def quantize_with_multiplier(x, m, fmt: Fmt) -> np.ndarray:
    x = _c32(x)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().or_quantize_with_multiplier(_p(x, _f32p), x.size, float(F32(m)), fmt.fid, _p(out, _u8p))
    return out


def dequantize(codes, s, fmt: Fmt) -> np.ndarray:
    c = _cu8(codes)
    out = np.empty(c.shape, dtype=np.float32)
    lib().or_dequantize(_p(c, _u8p), c.size, float(F32(s)), fmt.fid, _p(out, _f32p))
    return out


def quantize_tensor(x, fmt: Fmt, amax=None):
    x = _c32(x)
    codes = np.empty(x.shape, dtype=np.uint8)
    s, a = ctypes.c_float(), ctypes.c_float()
    _, ap = _opt32(amax)
    if lib().or_quantize_tensor(_p(x, _f32p), x.size, fmt.fid, ap, _p(codes, _u8p), ctypes.byref(s),
                                ctypes.byref(a)):
        raise NonFinite("non-finite element")
    return codes, F32(s.value), F32(a.value)


BLOCK = 128
BLOCK1D = 512


def block_grid(d_out, d_in, b=BLOCK):
    return (d_out + b - 1) // b, (d_in + b - 1) // b


def block_amax(x, b=BLOCK) -> np.ndarray:
    x = _c32(x)
    out = np.empty(block_grid(*x.shape, b), dtype=np.float32)
    if lib().or_block_amax(_p(x, _f32p), x.shape[0], x.shape[1], b, _p(out, _f32p)):
        raise NonFinite("non-finite element")
    return out


def quantize_block128(x, fmt: Fmt, amax=None):
    x = _c32(x)
    d_out, d_in = x.shape
    nb = block_grid(d_out, d_in)
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(nb, dtype=np.float32)
    am = np.empty(nb, dtype=np.float32)
    _, ap = _opt32(amax)
    if lib().or_quantize_block2d(_p(x, _f32p), d_out, d_in, BLOCK, fmt.fid, ap, _p(codes, _u8p),
                                 _p(scales, _f32p), _p(am, _f32p)):
        raise NonFinite("non-finite element")
    return codes, scales, am


def dequantize_block128(codes, scales, fmt: Fmt) -> np.ndarray:
    c = _cu8(codes)
    s = _c32(scales)
    out = np.empty(c.shape, dtype=np.float32)
    lib().or_dequantize_block2d(_p(c, _u8p), c.shape[0], c.shape[1], BLOCK, _p(s, _f32p), fmt.fid, _p(out, _f32p))
    return out


def quantize_block1d(x, fmt: Fmt, amax=None, b=BLOCK1D):
    x = _c32(x)
    n = x.size
    nb = (n + b - 1) // b
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(nb, dtype=np.float32)
    am = np.empty(nb, dtype=np.float32)
    _, ap = _opt32(amax)
    if lib().or_quantize_block1d(_p(x, _f32p), n, b, fmt.fid, ap, _p(codes, _u8p), _p(scales, _f32p),
                                 _p(am, _f32p)):
        raise NonFinite("non-finite element")
    return codes, scales, am


def dequantize_block1d(codes, scales, fmt: Fmt, b=BLOCK1D) -> np.ndarray:
    c = _cu8(codes)
    s = _c32(scales)
    out = np.empty(c.shape, dtype=np.float32)
    lib().or_dequantize_block1d(_p(c, _u8p), c.size, b, _p(s, _f32p), fmt.fid, _p(out, _f32p))
    return out


def quantize_nvfp4(x, amax=None):
    x = _c32(x)
    d_out, d_in = x.shape
    if d_in % 16:
        raise ValueError("NVFP4 needs d_in to be a multiple of 16")
    packed = np.empty((d_out, d_in // 2), dtype=np.uint8)
    bs = np.empty((d_out, d_in // 16), dtype=np.uint8)
    st, at = ctypes.c_float(), ctypes.c_float()
    _, ap = _opt32(amax)
    if lib().or_quantize_nvfp4(_p(x, _f32p), d_out, d_in, ap, _p(packed, _u8p), _p(bs, _u8p), ctypes.byref(st),
                               ctypes.byref(at)):
        raise NonFinite("non-finite element")
    return packed, bs, F32(st.value), F32(at.value)


def dequantize_nvfp4(packed, block_scales, s_t) -> np.ndarray:
    p = _cu8(packed)
    bs = _cu8(block_scales)
    d_out, d_in = p.shape[0], p.shape[1] * 2
    out = np.empty((d_out, d_in), dtype=np.float32)
    lib().or_dequantize_nvfp4(_p(p, _u8p), _p(bs, _u8p), float(F32(s_t)), d_out, d_in, _p(out, _f32p))
    return out


def quantize(x, fmt: str, scaling: str = "tensor", amax=None):
    """Returns a dict with 'codes', 'scales', 'tensor_scale' (NVFP4) and 'amax', as the numpy
    statement does."""
    if fmt == "f32":
        return {"codes": _c32(x).copy(), "scales": None, "tensor_scale": None, "amax": None}
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
        return _c32(q["codes"])
    if fmt == "nvfp4":
        return dequantize_nvfp4(q["codes"], q["scales"], q["tensor_scale"])
    f = FORMATS[fmt]
    if scaling == "tensor":
        return dequantize(q["codes"], q["scales"][0], f)
    if scaling == "block512":
        return dequantize_block1d(q["codes"], q["scales"], f)
    return dequantize_block128(q["codes"], q["scales"], f)


def replica_reduce(qs, fmt: str, scaling: str = "tensor") -> np.ndarray:
    """(deq_0 + ... + deq_{R-1}) / R with FP32 additions in replica order."""
    deq = np.stack([dequantize_any(q, fmt, scaling) for q in qs]).astype(np.float32)
    out = np.empty(deq.shape[1:], dtype=np.float32)
    deq = np.ascontiguousarray(deq)
    lib().or_replica_mean(_p(deq, _f32p), deq.shape[0], out.size, _p(out, _f32p))
    return out


def boundary_hits(x, fmt: str, scaling: str = "tensor"):
    x = _c32(x)
    q = quantize(x, fmt, scaling)
    c = _cu8(q["codes"])
    counts = np.zeros(3, dtype=np.uint64)
    lib().or_boundary_counts(_p(x, _f32p), _p(c, _u8p), x.size, FORMATS[fmt].fid, _p(counts, _u64p))
    return int(counts[0]), int(counts[1]), int(counts[2])


def window_scores(counts):
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.uint64).reshape(-1, 3))
    out = np.empty(c.shape[0], dtype=np.float64)
    lib().or_window_scores(_p(c, _u64p), c.shape[0], _p(out, _f64p))
    return [float(v) for v in out]


def fragility_score(hits) -> float:
    return window_scores([hits])[0]


def _ranked(scores):
    s = _c64(scores)
    order = np.empty(s.size, dtype=np.int32)
    lib().or_rank_layers(_p(s, _f64p), s.size, _p(order, _i32p))
    return [int(i) for i in order]


def select_fragile(scores, k):
    return _ranked(scores)[:k]


def knee_count(ranked, k_min=1, k_max=None):
    r = _c64(ranked)
    L = r.size
    k = lib().or_knee_count(_p(r, _f64p), L, k_min, L if k_max is None else k_max)
    if k < 0:
        raise ValueError("need 1 <= k_min <= k_max <= number of layers")
    return int(k)


def select_fragile_knee(scores, k_min=1, k_max=None):
    order = _ranked(scores)
    k = knee_count([scores[i] for i in order], k_min, k_max)
    return order[:k]


# ---- K-FAC factors, Cholesky, triangular solves -------------------------------------------

def kfac_factor(a) -> np.ndarray:
    a = _c64(a)
    T, d = a.shape
    out = np.empty((d, d), dtype=np.float64)
    lib().or_kfac_factor(_p(a, _f64p), T, d, _p(out, _f64p))
    return out


def cholesky(A) -> np.ndarray:
    A = _c64(A)
    L = np.empty_like(A)
    piv = lib().or_cholesky(_p(A, _f64p), A.shape[0], _p(L, _f64p))
    if piv >= 0:
        raise NotPositiveDefinite(f"pivot {piv}")
    return L


def lower_inverse(L) -> np.ndarray:
    L = _c64(L)
    X = np.empty_like(L)
    lib().or_lower_inverse(_p(L, _f64p), L.shape[0], _p(X, _f64p))
    return X


def solve_right_lower_t(W, L) -> np.ndarray:
    W, L = _c64(W), _c64(L)
    X = np.empty_like(W)
    lib().or_solve_right_lower_t(_p(W, _f64p), _p(L, _f64p), W.shape[0], W.shape[1], _p(X, _f64p))
    return X


def solve_left_lower(L, W) -> np.ndarray:
    W, L = _c64(W), _c64(L)
    Y = np.empty_like(W)
    lib().or_solve_left_lower(_p(L, _f64p), _p(W, _f64p), W.shape[0], W.shape[1], _p(Y, _f64p))
    return Y


def _matmul(A, B) -> np.ndarray:
    A, B = _c64(A), _c64(B)
    out = np.empty((A.shape[0], B.shape[1]), dtype=np.float64)
    lib().or_matmul(_p(A, _f64p), _p(B, _f64p), A.shape[0], A.shape[1], B.shape[1], _p(out, _f64p))
    return out


def _matmul_bt(A, B) -> np.ndarray:
    A, B = _c64(A), _c64(B)
    out = np.empty((A.shape[0], B.shape[0]), dtype=np.float64)
    lib().or_matmul_bt(_p(A, _f64p), _p(B, _f64p), A.shape[0], A.shape[1], B.shape[0], _p(out, _f64p))
    return out


# ---- eigen solvers --------------------------------------------------------------------------

def jacobi_eigh(S, tol=1e-15, max_sweeps=40):
    S = _c64(S)
    n = S.shape[0]
    w = np.empty(n, dtype=np.float64)
    V = np.empty((n, n), dtype=np.float64)
    lib().or_jacobi_eigh(_p(S, _f64p), n, tol, max_sweeps, _p(w, _f64p), _p(V, _f64p))
    return w, V


def _omega(n, k, seed):
    # the Gaussian start of the numpy statement (the same generator and seed), passed in
    return _c64(np.random.default_rng(seed).standard_normal((n, k)))


def _subspace(mode, M, T, n, k, iters, seed, apply_A=None):
    om = _omega(n, k, seed)
    mu = np.empty(k, dtype=np.float64)
    U = np.empty((n, k), dtype=np.float64)
    keep = []

    def cb(xp, nn, kk, yp, _user):
        X = np.ctypeslib.as_array(xp, shape=(nn, kk))
        Y = np.ctypeslib.as_array(yp, shape=(nn, kk))
        Y[:] = apply_A(X.copy())

    fn = APPLY_FN(cb) if apply_A is not None else APPLY_FN()
    keep.append(fn)
    Mp = _p(M, _f64p) if M is not None else None
    lib().or_subspace_iteration(mode, Mp, T, n, k, iters, _p(om, _f64p), fn, None, _p(mu, _f64p), _p(U, _f64p))
    return mu, U


def subspace_iteration(apply_A, n, k=64, iters=16, seed=12345):
    """Top-k Ritz pairs of the operator apply_A (a callable X -> A X, or an explicit n x n
    matrix)."""
    if callable(apply_A):
        return _subspace(2, None, 0, n, k, iters, seed, apply_A)
    return _subspace(0, _c64(apply_A), 0, n, k, iters, seed)


class LowRankFactor:
    """A ~ U diag(mu - sigma) U^T + sigma I; mu the top-r eigenvalues of A."""

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
        out = np.empty((d, d), dtype=np.float64)
        U, mu = _c64(self.U), _c64(self.mu)
        lib().or_lowrank_dense(_p(U, _f64p), _p(mu, _f64p), d, self.rank, self.sigma, _p(out, _f64p))
        return out


def lowrank_from_eigs(mu_all, V_all, trace, d_in, r) -> LowRankFactor:
    mu_all, V_all = _c64(mu_all), _c64(V_all)
    U = np.empty((d_in, r), dtype=np.float64)
    mu = np.empty(r, dtype=np.float64)
    sig = ctypes.c_double()
    if lib().or_lowrank_from_eigs(_p(mu_all, _f64p), _p(V_all, _f64p), V_all.shape[1], float(trace), d_in, r,
                                  _p(U, _f64p), _p(mu, _f64p), ctypes.byref(sig)):
        raise NotPositiveDefinite(f"sigma = {sig.value}, min mu = {np.min(mu)}")
    return LowRankFactor(U, mu, sig.value)


def lowrank_factor_from_A(A, r=32, k=64, iters=16, seed=12345) -> LowRankFactor:
    """Rank-r factor of an explicit A: exact Jacobi when d <= 128, else subspace iteration."""
    A = _c64(A)
    d = A.shape[0]
    tr = float(lib().or_trace(_p(A, _f64p), d))
    if d <= 128:
        mu, V = jacobi_eigh(A)
    else:
        mu, V = _subspace(0, A, 0, d, min(k, d), iters, seed)
    return lowrank_from_eigs(mu, V, tr, d, r)


def lowrank_factor_from_activations(a, r=32, k=64, iters=16, seed=12345) -> LowRankFactor:
    """Rank-r factor of A = a^T a / T without forming A when d > 128."""
    a = _c64(a)
    T, d = a.shape
    if d <= 128:
        return lowrank_factor_from_A(kfac_factor(a), r=r)
    tr = float(lib().or_activation_trace(_p(a, _f64p), T, d))
    mu, V = _subspace(1, a, T, d, min(k, d), iters, seed)
    return lowrank_from_eigs(mu, V, tr, d, r)


def _lowrank_apply(W, F: LowRankFactor, inverse):
    W = _c64(W)
    U, mu = _c64(F.U), _c64(F.mu)
    out = np.empty_like(W)
    lib().or_lowrank_apply(_p(W, _f64p), W.shape[0], W.shape[1], _p(U, _f64p), _p(mu, _f64p), F.rank, F.sigma,
                           int(inverse), _p(out, _f64p))
    return out


def lowrank_T(F: LowRankFactor, inverse=False) -> np.ndarray:
    d = F.U.shape[0]
    U, mu = _c64(F.U), _c64(F.mu)
    out = np.empty((d, d), dtype=np.float64)
    lib().or_lowrank_T(_p(U, _f64p), _p(mu, _f64p), d, F.rank, F.sigma, int(inverse), _p(out, _f64p))
    return out


def lowrank_whiten(W, F: LowRankFactor) -> np.ndarray:
    return _lowrank_apply(W, F, False)


def lowrank_unwhiten(X, F: LowRankFactor) -> np.ndarray:
    return _lowrank_apply(X, F, True)


def chol_input_whiten(W, LA) -> np.ndarray:
    return solve_right_lower_t(W, LA)


def chol_two_sided_whiten(W, LG, LA) -> np.ndarray:
    return solve_right_lower_t(solve_left_lower(LG, W), LA)


def chol_input_unwhiten(X, LA) -> np.ndarray:
    return _matmul_bt(X, LA)


def chol_two_sided_unwhiten(X, LG, LA) -> np.ndarray:
    return _matmul_bt(_matmul(LG, X), LA)


def chol_whiten_with_inverses(W, LAinv, LGinv=None) -> np.ndarray:
    X = _matmul_bt(W, LAinv)
    if LGinv is not None:
        X = _matmul(LGinv, X)
    return X


class Xform:
    """A transform: kind in {identity, lowrank, chol_input, chol_two_sided} and its factor."""

    def __init__(self, kind, F=None, LA=None, LG=None, LAinv=None, LGinv=None):
        self.kind, self.F, self.LA, self.LG = kind, F, LA, LG
        self.LAinv, self.LGinv = LAinv, LGinv

    def whiten(self, W):
        if self.kind == "identity":
            return _c64(W)
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
            return _c64(X)
        if self.kind == "lowrank":
            return lowrank_unwhiten(X, self.F)
        if self.kind == "chol_input":
            return chol_input_unwhiten(X, self.LA)
        return chol_two_sided_unwhiten(X, self.LG, self.LA)


def _round_f32(x) -> np.ndarray:
    x = _c64(x)
    out = np.empty(x.shape, dtype=np.float32)
    lib().or_round_f32(_p(x, _f64p), x.size, _p(out, _f32p))
    return out


def _binop(fn, a, b):
    a, b = _c32(a), _c32(b)
    out = np.empty(a.shape, dtype=np.float32)
    fn(_p(a, _f32p), _p(b, _f32p), a.size, _p(out, _f32p))
    return out


def encode_layer(W, xf: Xform, fmt: str, scaling="tensor", amax=None, residual=None):
    """Whiten, optionally add the error-feedback residual, scale and quantise (Algorithm 1).
    Returns (q, transformed FP32, new residual or None)."""
    Wt = _round_f32(xf.whiten(W))
    if residual is not None:
        Wt = _binop(lib().or_add_f32, Wt, residual)
    q = quantize(Wt, fmt, scaling, amax)
    new_res = None
    if residual is not None:
        new_res = _binop(lib().or_sub_f32, Wt, dequantize_any(q, fmt, scaling))
    return q, Wt, new_res


def decode_layer(X, xf: Xform) -> np.ndarray:
    return xf.unwhiten(X)


def fidelity(g_hat, g):
    gh, gg = _c64(np.ravel(g_hat)), _c64(np.ravel(g))
    out = np.empty(4, dtype=np.float64)
    lib().or_fidelity(_p(gh, _f64p), _p(gg, _f64p), gh.size, _p(out, _f64p))
    return {"rel_l2": float(out[0]), "cos": float(out[1]), "max_err": float(out[2]), "mse": float(out[3])}


def toy_quantize(v):
    v = _c64(v)
    out = np.empty_like(v)
    lib().or_toy_quantize(_p(v, _f64p), v.size, _p(out, _f64p))
    return out


_init_formats()
