"""Thin Python binding of libgift (ctypes).

Every function here has the name of the C entry point it wraps and only marshals
arguments: torch tensors become device pointers, None becomes NULL, the current
torch stream becomes the cudaStream_t.  All arithmetic runs in libgift's CUDA
kernels; nothing in this module computes on tensor data.  If libgift.so is not
built, the first call raises RuntimeError (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgift.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "gift.h")

# ---- enums (values fixed by include/gift.h) ---------------------------------------------
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NONFINITE, ERR_NOT_PD, ERR_TIMEOUT, ERR_NOT_CONVERGED = range(8)
FMT = {"f32": 0, "e4m3": 1, "e5m2": 2, "nvfp4": 3}
SCALING = {"tensor": 0, "block128": 1, "block512": 2}
XFORM = {"identity": 0, "lowrank": 1, "chol_input": 2, "chol_two_sided": 3}
PREC = {"fp32": 0, "tc": 1}
DTYPE = {"f32": 0, "bf16": 1}
OP = {"factor_update": 0, "encode": 1, "decode": 2, "amax": 3, "kfac_factor": 4, "reduce_decode": 5}
OPT_SUBSPACE_ITERS = 0
OPT_BARRIER_WAIT = 1
OPT_SKETCH = 2
OPT_SMS = 3

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


class GiftFactor(ctypes.Structure):
    _fields_ = [("kind", _i), ("d_in", _i), ("d_out", _i), ("rank", _i),
                ("U", _vp), ("mu", _vp), ("sigma", _vp),
                ("LA", _vp), ("LAinv", _vp), ("LG", _vp), ("LGinv", _vp), ("planes", _vp)]


class GiftError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {status_string(status)} ({status})"
        if status == ERR_CUDA:
            msg += f": {lib().gift_last_error().decode()}"
        super().__init__(msg)
        self.status = status


_LIB = None


def _declare(lib):
    sig = {
        "gift_create": (_i, [ctypes.POINTER(_vp), _i]),
        "gift_destroy": (None, [_vp]),
        "gift_set_option": (_i, [_vp, _i, ctypes.c_longlong]),
        "gift_status_string": (ctypes.c_char_p, [_i]),
        "gift_version": (_i, []),
        "gift_last_error": (ctypes.c_char_p, []),
        "gift_workspace_bytes": (_sz, [_vp, _i, _i, _i, _i, _i, _i, _i, _i]),
        "gift_code_sizes": (_i, [_i, _i, _i, _i, ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
        "gift_factor_update": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _i, _i, _vp, _i, ctypes.c_uint64, _i,
                                    _vp, _sz, _vp, _vp]),
        "gift_factor_update_from_kfac": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _vp, ctypes.c_uint64, _i, _vp,
                                              _sz, _vp, _vp]),
        "gift_kfac_factor": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp, _vp]),
        "gift_boundary_hit_rates": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_i), ctypes.POINTER(_i), _i,
                                         _i, _vp, _vp, _sz, _vp, _vp]),
        "gift_factor_planes_bytes": (_sz, [_i]),
        "gift_factor_prepare": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp]),
        "gift_amax": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp, _vp]),
        "gift_encode": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                             _vp, _vp, _sz, _vp, _vp]),
        "gift_encode_replicas": (_i, [_vp, ctypes.POINTER(GiftFactor), _i, ctypes.POINTER(_vp), _i, _i, _i, _i, _i,
                                      ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                      ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, _sz, _vp, _vp]),
        "gift_amax_replicas": (_i, [_vp, ctypes.POINTER(GiftFactor), _i, ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _vp,
                                    _vp, _sz, _vp, _vp]),
        "gift_encode_replicas_shared": (_i, [_vp, ctypes.POINTER(GiftFactor), _i, ctypes.POINTER(_vp), _i, _i, _i, _i,
                                             _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp,
                                             _vp, _sz, _vp, _vp]),
        "gift_select_fragile": (_i, [_i, _vp, _i, _i, _i, _vp, _vp, _vp]),
        "gift_replica_reduce": (_i, [_vp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i, _i,
                                     _i, _i, _vp, _vp, _vp]),
        "gift_decode": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz,
                             _vp, _vp]),
        "gift_reduce_decode": (_i, [_vp, ctypes.POINTER(GiftFactor), _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                    ctypes.POINTER(_vp), _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _vp, _vp]),
        "gift_boundary_hit_rate": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp, _vp]),
        "gift_encode_lowrank_noalloc": (_i, [_vp, ctypes.POINTER(GiftFactor), _vp, _i, _i, _i, _vp, _vp, _vp, _vp,
                                             _vp, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args


def lib():
    """The loaded libgift (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgift is not built ({LIB_PATH} missing); run fac_whitening_gb300.build.build()")
        _LIB = ctypes.CDLL(LIB_PATH)
        _declare(_LIB)
    return _LIB


def header_functions():
    """Names of every function declared in include/gift.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_ ]+\*?\s*\*?(gift_[a-z0-9_]+)\s*\(", text, re.M)))


def _p(t) -> Optional[int]:
    """Address of a caller buffer for the library: None, a raw device address (int), or a
    contiguous CUDA tensor.  A host tensor or a strided view is refused here, since a kernel
    would read it as contiguous device memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not getattr(t, "is_cuda", False):
        raise ValueError("libgift buffers live in device memory: pass a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("libgift buffers are dense row-major: pass a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str):
    if status != OK:
        raise GiftError(status, where)


def status_string(status: int) -> str:
    return lib().gift_status_string(status).decode()


def gift_version() -> int:
    return lib().gift_version()


# ---- context ------------------------------------------------------------------------------
class Context:
    """Owns one gift_ctx for a CUDA device."""

    def __init__(self, device: int = 0):
        h = _vp()
        _check(lib().gift_create(ctypes.byref(h), device), "gift_create")
        self.handle = h
        self.device = device

    def close(self):
        if self.handle:
            lib().gift_destroy(self.handle)
            self.handle = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gift_create(device: int = 0) -> Context:
    return Context(device)


def gift_set_option(ctx: Context, opt: int, value: int):
    _check(lib().gift_set_option(ctx.handle, opt, value), "gift_set_option")


def gift_workspace_bytes(ctx: Context, op: str, kind: str, fmt: str, scaling: str, d_out: int, d_in: int,
                         T: int = 0, rank: int = 32) -> int:
    n = lib().gift_workspace_bytes(ctx.handle, OP[op], XFORM[kind], FMT[fmt], SCALING[scaling], d_out, d_in, T, rank)
    if n == ctypes.c_size_t(-1).value:
        raise GiftError(ERR_INVALID_ARG, "gift_workspace_bytes")
    return n


def gift_code_sizes(fmt: str, scaling: str, d_out: int, d_in: int):
    cb, sc = _sz(), _sz()
    _check(lib().gift_code_sizes(FMT[fmt], SCALING[scaling], d_out, d_in, ctypes.byref(cb), ctypes.byref(sc)),
           "gift_code_sizes")
    return cb.value, sc.value


def gift_select_fragile(counts, k: int = 0, k_min: int = 1, k_max: Optional[int] = None):
    """Host-side layer selection from window counts (L x 3: upper, lower, n per layer).
    Returns (order, scores, k): layer indices by descending score, the scores, and how many
    of order are selected (k > 0: that many; k = 0: at the knee within [k_min, k_max])."""
    flat = [int(v) for row in counts for v in row]
    L = len(flat) // 3
    if L * 3 != len(flat):
        raise ValueError("counts must be L rows of (upper, lower, n)")
    c = (ctypes.c_ulonglong * max(len(flat), 1))(*flat)
    order = (ctypes.c_int * max(L, 1))()
    scores = (ctypes.c_double * max(L, 1))()
    k_out = ctypes.c_int()
    _check(lib().gift_select_fragile(L, ctypes.cast(c, _vp), k, k_min, L if k_max is None else k_max,
                                     ctypes.cast(order, _vp), ctypes.cast(scores, _vp), ctypes.byref(k_out)),
           "gift_select_fragile")
    return list(order)[:L], list(scores)[:L], k_out.value


# ---- factor -------------------------------------------------------------------------------
@dataclass
class Factor:
    """Device buffers of one layer's factor (torch tensors owned by the caller)."""
    kind: str
    d_out: int
    d_in: int
    rank: int = 32
    U: object = None
    mu: object = None
    sigma: object = None
    LA: object = None
    LAinv: object = None
    LG: object = None
    LGinv: object = None
    planes: object = None

    @staticmethod
    def empty(kind: str, d_out: int, d_in: int, rank: int = 32, device="cuda", planes: bool = False) -> "Factor":
        """Zeroed factor buffers; planes=True also allocates the cached U term planes (LOWRANK)."""
        import torch
        f = Factor(kind, d_out, d_in, rank)
        z = lambda *s: torch.zeros(*s, dtype=torch.float32, device=device)  # noqa: E731
        if kind == "lowrank":
            f.U, f.mu, f.sigma = z(d_in, rank), z(rank), z(1)
            if planes:
                f.planes = torch.zeros(lib().gift_factor_planes_bytes(d_in), dtype=torch.uint8, device=device)
        elif kind in ("chol_input", "chol_two_sided"):
            f.LA, f.LAinv = z(d_in, d_in), z(d_in, d_in)
            if kind == "chol_two_sided":
                f.LG, f.LGinv = z(d_out, d_out), z(d_out, d_out)
        return f

    def c_struct(self) -> GiftFactor:
        return GiftFactor(XFORM[self.kind], self.d_in, self.d_out, self.rank, _p(self.U), _p(self.mu),
                          _p(self.sigma), _p(self.LA), _p(self.LAinv), _p(self.LG), _p(self.LGinv), _p(self.planes))


def _fptr(f: Optional[Factor]):
    if f is None:
        return None
    return ctypes.byref(f.c_struct())


def gift_factor_update(ctx: Context, f: Factor, a, delta=None, seed: int = 0, prec: str = "fp32", ws=None,
                       status=None, stream=None):
    import torch
    a_dt = DTYPE["bf16"] if a.dtype == torch.bfloat16 else DTYPE["f32"]
    d_dt = DTYPE["bf16"] if (delta is not None and delta.dtype == torch.bfloat16) else DTYPE["f32"]
    st = f.c_struct()
    _check(lib().gift_factor_update(ctx.handle, ctypes.byref(st), _p(a), a_dt, a.shape[0], _p(delta), d_dt,
                                    seed, PREC[prec], _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                    _p(status), _stream(stream)), "gift_factor_update")


def gift_factor_update_from_kfac(ctx: Context, f: Factor, A, G=None, seed: int = 0, prec: str = "fp32", ws=None,
                                 status=None, stream=None):
    st = f.c_struct()
    _check(lib().gift_factor_update_from_kfac(ctx.handle, ctypes.byref(st), _p(A), _p(G), seed, PREC[prec], _p(ws),
                                              0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                              _stream(stream)), "gift_factor_update_from_kfac")


def gift_factor_prepare(ctx: Context, f: Factor, stream=None):
    st = f.c_struct()
    _check(lib().gift_factor_prepare(ctx.handle, ctypes.byref(st), _stream(stream)), "gift_factor_prepare")


def gift_kfac_factor(ctx: Context, a, A_out, prec: str = "fp32", ws=None, status=None, stream=None):
    import torch
    a_dt = DTYPE["bf16"] if a.dtype == torch.bfloat16 else DTYPE["f32"]
    T, d = a.shape
    _check(lib().gift_kfac_factor(ctx.handle, _p(a), a_dt, T, d, PREC[prec], _p(A_out), _p(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(), _p(status), _stream(stream)),
           "gift_kfac_factor")


def gift_amax(ctx: Context, f: Optional[Factor], W, fmt: str, scaling: str, amax_accum, residual=None,
              prec: str = "fp32", ws=None, status=None, stream=None):
    d_out, d_in = W.shape
    _check(lib().gift_amax(ctx.handle, _fptr(f), _p(W), d_out, d_in, FMT[fmt], SCALING[scaling], PREC[prec],
                           _p(residual), _p(amax_accum), _p(ws),
                           0 if ws is None else ws.numel() * ws.element_size(), _p(status), _stream(stream)),
           "gift_amax")


def gift_encode(ctx: Context, f: Optional[Factor], W, fmt: str, scaling: str, codes, scales=None,
                tensor_scale=None, amax_in=None, residual=None, transformed_out=None, amax_out=None,
                prec: str = "fp32", ws=None, status=None, stream=None):
    d_out, d_in = W.shape
    _check(lib().gift_encode(ctx.handle, _fptr(f), _p(W), d_out, d_in, FMT[fmt], SCALING[scaling], PREC[prec],
                             _p(amax_in), _p(residual), _p(codes), _p(scales), _p(tensor_scale),
                             _p(transformed_out), _p(amax_out), _p(ws),
                             0 if ws is None else ws.numel() * ws.element_size(), _p(status), _stream(stream)),
           "gift_encode")


def gift_encode_replicas(ctx: Context, f: Optional[Factor], Ws: Sequence, fmt: str, scaling: str, codes: Sequence,
                         scales: Optional[Sequence] = None, tensor_scales: Optional[Sequence] = None,
                         amax_in: Optional[Sequence] = None, amax_out: Optional[Sequence] = None,
                         prec: str = "fp32", ws=None, status=None, stream=None):
    R = len(Ws)
    d_out, d_in = Ws[0].shape
    arr = lambda xs: (_vp * R)(*[_p(x) for x in xs]) if xs is not None else None  # noqa: E731
    _check(lib().gift_encode_replicas(ctx.handle, _fptr(f), R, arr(Ws), d_out, d_in, FMT[fmt], SCALING[scaling],
                                      PREC[prec], arr(amax_in), arr(codes), arr(scales), arr(tensor_scales),
                                      arr(amax_out), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                      _p(status), _stream(stream)), "gift_encode_replicas")


def gift_encode_replicas_shared(ctx: Context, f: Optional[Factor], Ws: Sequence, fmt: str, scaling: str,
                                codes: Sequence, scales: Sequence, tensor_scales: Optional[Sequence] = None,
                                shared_amax_out=None, prec: str = "fp32", ws=None, status=None, stream=None):
    R = len(Ws)
    d_out, d_in = Ws[0].shape
    arr = lambda xs: (_vp * R)(*[_p(x) for x in xs]) if xs is not None else None  # noqa: E731
    _check(lib().gift_encode_replicas_shared(ctx.handle, _fptr(f), R, arr(Ws), d_out, d_in, FMT[fmt],
                                             SCALING[scaling], PREC[prec], arr(codes), arr(scales),
                                             arr(tensor_scales), _p(shared_amax_out), _p(ws),
                                             0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                             _stream(stream)), "gift_encode_replicas_shared")


def gift_amax_replicas(ctx: Context, f: Optional[Factor], Ws: Sequence, fmt: str, scaling: str, amax_accum,
                       prec: str = "fp32", ws=None, status=None, stream=None):
    R = len(Ws)
    d_out, d_in = Ws[0].shape
    _check(lib().gift_amax_replicas(ctx.handle, _fptr(f), R, (_vp * R)(*[_p(W) for W in Ws]), d_out, d_in, FMT[fmt],
                                    SCALING[scaling], PREC[prec], _p(amax_accum), _p(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                    _stream(stream)), "gift_amax_replicas")


def gift_replica_reduce(ctx: Context, codes: Sequence, scales: Optional[Sequence], fmt: str, scaling: str,
                        d_out: int, d_in: int, avg_out, tensor_scales: Optional[Sequence] = None, status=None,
                        stream=None):
    R = len(codes)
    arr = lambda xs: (_vp * R)(*[_p(x) for x in xs]) if xs is not None else None  # noqa: E731
    _check(lib().gift_replica_reduce(ctx.handle, R, arr(codes), arr(scales), arr(tensor_scales), FMT[fmt],
                                     SCALING[scaling], d_out, d_in, _p(avg_out), _p(status), _stream(stream)),
           "gift_replica_reduce")


def gift_reduce_decode(ctx: Context, f: Optional[Factor], codes: Sequence, scales: Optional[Sequence], fmt: str,
                       scaling: str, d_out: int, d_in: int, W_out, avg_out=None, tensor_scales=None,
                       prec: str = "fp32", ws=None, status=None, stream=None):
    R = len(codes)
    arr = lambda xs: (_vp * R)(*[_p(x) for x in xs]) if xs is not None else None  # noqa: E731
    _check(lib().gift_reduce_decode(ctx.handle, _fptr(f), R, arr(codes), arr(scales), arr(tensor_scales), FMT[fmt],
                                    SCALING[scaling], PREC[prec], d_out, d_in, _p(avg_out), _p(W_out), _p(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                    _stream(stream)), "gift_reduce_decode")


def gift_decode(ctx: Context, f: Optional[Factor], inp, in_is_codes: bool, fmt: str, scaling: str, d_out: int,
                d_in: int, W_out, scales=None, tensor_scale=None, prec: str = "fp32", ws=None, status=None,
                stream=None):
    _check(lib().gift_decode(ctx.handle, _fptr(f), _p(inp), int(bool(in_is_codes)), _p(scales), _p(tensor_scale),
                             FMT[fmt], SCALING[scaling], PREC[prec], d_out, d_in, _p(W_out), _p(ws),
                             0 if ws is None else ws.numel() * ws.element_size(), _p(status), _stream(stream)),
           "gift_decode")


def gift_boundary_hit_rate(ctx: Context, W, fmt: str, scaling: str, counts, ws=None, status=None, stream=None):
    d_out, d_in = W.shape
    _check(lib().gift_boundary_hit_rate(ctx.handle, _p(W), d_out, d_in, FMT[fmt], SCALING[scaling], _p(counts),
                                        _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                        _stream(stream)), "gift_boundary_hit_rate")


def gift_boundary_hit_rates(ctx: Context, Ws: Sequence, fmt: str, scaling: str, counts, ws=None, status=None,
                            stream=None):
    """Hit counts of several tensors in one call; counts is an n x 3 int64 device tensor."""
    n = len(Ws)
    ptrs = (_vp * n)(*[_p(W) for W in Ws])
    rows = (_i * n)(*[int(W.shape[0]) for W in Ws])
    cols = (_i * n)(*[int(W.shape[1]) for W in Ws])
    _check(lib().gift_boundary_hit_rates(ctx.handle, n, ptrs, rows, cols, FMT[fmt], SCALING[scaling], _p(counts),
                                         _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(status),
                                         _stream(stream)), "gift_boundary_hit_rates")


def gift_encode_lowrank_noalloc(ctx: Context, f: Factor, W, fmt: str, codes, scales, amax_in=None, amax_out=None,
                                status=None, stream=None):
    """Rank-r encode without a workspace (scratch lives inside the library; see gift.h)."""
    d_out, d_in = W.shape
    _check(lib().gift_encode_lowrank_noalloc(ctx.handle, _fptr(f), _p(W), d_out, d_in, FMT[fmt], _p(amax_in),
                                             _p(codes), _p(scales), _p(amax_out), _p(status), _stream(stream)),
           "gift_encode_lowrank_noalloc")
