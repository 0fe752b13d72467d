"""Helpers for the GPU parity tests: run libgift entry points on numpy inputs and
return numpy outputs.  (Marshalling only; the comparisons live in the tests.)"""
import numpy as np
import torch

from fac_whitening_gb300 import gift as G

DEV = torch.device("cuda")
_CTX = None


def ctx():
    global _CTX
    if _CTX is None:
        _CTX = G.Context(torch.cuda.current_device())
    return _CTX


def t(x, dtype=torch.float32):
    return torch.as_tensor(np.ascontiguousarray(x)).to(device=DEV, dtype=dtype)


def status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def ws(op, kind, fmt, scaling, d_out, d_in):
    n = G.gift_workspace_bytes(ctx(), op, kind, fmt, scaling, d_out, d_in)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=DEV)


def alloc_codes(fmt, scaling, d_out, d_in):
    cb, sc = G.gift_code_sizes(fmt, scaling, d_out, d_in)
    if fmt == "f32":
        return torch.empty(d_out, d_in, dtype=torch.float32, device=DEV), None, None
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    if fmt == "nvfp4":
        return codes, torch.empty(sc, dtype=torch.uint8, device=DEV), torch.empty(1, dtype=torch.float32, device=DEV)
    return codes, torch.empty(sc, dtype=torch.float32, device=DEV), None


def factor_to_gpu(kind, d_out, d_in, F=None, LA=None, LAinv=None, LG=None, LGinv=None, rank=32):
    if kind == "lowrank":
        return G.Factor("lowrank", d_out, d_in, F.rank, U=t(F.U), mu=t(F.mu), sigma=t([F.sigma]))
    f = G.Factor(kind, d_out, d_in, rank, LA=t(LA), LAinv=t(LAinv))
    if kind == "chol_two_sided":
        f.LG, f.LGinv = t(LG), t(LGinv)
    return f


def encode(f, W, fmt, scaling="tensor", amax_in=None, residual=None, Wt=None, prec="fp32"):
    """Run gift_encode; returns a dict of numpy outputs (codes shaped like the oracle's)."""
    Wt = t(W) if Wt is None else Wt
    d_out, d_in = Wt.shape
    kind = "identity" if f is None else f.kind
    codes, scales, tscale = alloc_codes(fmt, scaling, d_out, d_in)
    tout = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    if scaling == "tensor" or fmt == "nvfp4":
        nam = 1
    elif scaling == "block512":
        nam = (d_out * d_in + 511) // 512
    else:
        nam = ((d_out + 127) // 128) * ((d_in + 127) // 128)
    amax_out = torch.empty(nam, dtype=torch.float32, device=DEV)
    R = None if residual is None else t(residual)
    st = status()
    G.gift_encode(ctx(), f, Wt, fmt, scaling, codes, scales, tscale,
                  amax_in=None if amax_in is None else t(np.atleast_1d(amax_in)),
                  residual=R, transformed_out=tout, amax_out=amax_out, prec=prec,
                  ws=ws("encode", kind, fmt, scaling, d_out, d_in), status=st)
    torch.cuda.synchronize()
    out = {"status": int(st.item()), "tout": tout.cpu().numpy(), "amax": amax_out.cpu().numpy()}
    if fmt == "f32":
        out["codes"] = codes.cpu().numpy()
    elif fmt == "nvfp4":
        out["codes"] = codes.cpu().numpy().reshape(d_out, d_in // 2)
        out["scales"] = scales.cpu().numpy().reshape(d_out, d_in // 16)
        out["tensor_scale"] = np.float32(tscale.item())
    else:
        out["codes"] = codes.cpu().numpy().reshape(d_out, d_in)
        sc = scales.cpu().numpy()
        out["scales"] = sc if scaling in ("tensor", "block512") else sc.reshape((d_out + 127) // 128, (d_in + 127) // 128)
    if R is not None:
        out["residual"] = R.cpu().numpy()
    out["_dev"] = (codes, scales, tscale)
    return out


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
