"""gift_reduce_decode: the replica reduce and the map back in one call ([notes] Algorithm 1:
AllReduceSum, Dequantize, divide by N, then multiply back with the factor; eq. (14)).

  - the average it can export (avg_out) is bit-identical to gift_replica_reduce's;
  - W_out is within 1e-5 (relative Frobenius, the FP32 path's tolerance) of the oracle's map
    back of that average, and equal to gift_decode applied to gift_replica_reduce's output;
  - rank-r, Cholesky and identity factors, FP8 / NVFP4 and block scaling, ragged shapes and a
    factor of rank below 32.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G

from gpu_util import DEV, alloc_codes, ctx, rel_fro, status, t, ws

pytestmark = pytest.mark.gpu


def rand_factor(d_out, d_in, seed, rank=32):
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((d_in, rank)))
    mu = np.sort(rng.uniform(0.5, 50.0, rank))[::-1].copy()
    F = O.LowRankFactor(U.astype(np.float32), mu.astype(np.float32), np.float32(0.05))
    return F, G.Factor("lowrank", d_out, d_in, rank, U=t(F.U), mu=t(F.mu), sigma=t([F.sigma]))


def encode_replicas(f, Ws, fmt, scaling, d_out, d_in):
    outs = [alloc_codes(fmt, scaling, d_out, d_in) for _ in Ws]
    st = status()
    kind = "identity" if f is None else f.kind
    G.gift_encode_replicas(ctx(), f, Ws, fmt, scaling, [o[0] for o in outs], scales=[o[1] for o in outs],
                           tensor_scales=[o[2] for o in outs] if fmt == "nvfp4" else None,
                           ws=ws("encode", kind, fmt, scaling, d_out, d_in), status=st)
    return [o[0] for o in outs], [o[1] for o in outs], ([o[2] for o in outs] if fmt == "nvfp4" else None)


def two_calls(f, codes, scales, tsc, fmt, scaling, d_out, d_in):
    kind = "identity" if f is None else f.kind
    avg = torch.empty(d_out, d_in, device=DEV)
    G.gift_replica_reduce(ctx(), codes, scales, fmt, scaling, d_out, d_in, avg, tensor_scales=tsc)
    ref = torch.empty(d_out, d_in, device=DEV)
    G.gift_decode(ctx(), f, avg, False, "f32", "tensor", d_out, d_in, ref,
                  ws=ws("decode", kind, "f32", "tensor", d_out, d_in))
    return avg, ref


@pytest.mark.parametrize("shape", [(1536, 6144), (1000, 4096), (384, 2112)], ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("fmt,R", [("e4m3", 8), ("e5m2", 3)])
def test_reduce_decode_matches_reduce_then_decode(shape, fmt, R):
    d_out, d_in = shape
    F, f = rand_factor(d_out, d_in, seed=51)
    gen = torch.Generator(device=DEV).manual_seed(52)
    Ws = [(torch.randn(d_out, d_in, generator=gen, device=DEV) * 0.1
           + (torch.randn(d_out, 32, generator=gen, device=DEV) * 3.0) @ f.U.T).contiguous() for _ in range(R)]
    codes, scales, _ = encode_replicas(f, Ws, fmt, "tensor", d_out, d_in)
    avg, ref = two_calls(f, codes, scales, None, fmt, "tensor", d_out, d_in)
    st = status()
    w = ws("reduce_decode", "lowrank", fmt, "tensor", d_out, d_in)
    for with_avg in (True, False):
        avg2 = torch.full((d_out, d_in), float("nan"), device=DEV) if with_avg else None
        out = torch.empty(d_out, d_in, device=DEV)
        G.gift_reduce_decode(ctx(), f, codes, scales, fmt, "tensor", d_out, d_in, out, avg_out=avg2, ws=w, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        if with_avg:
            assert torch.equal(avg2, avg)
        X = avg.cpu().numpy()
        assert rel_fro(out.cpu().numpy(), O.lowrank_unwhiten(X, F)) <= 1e-5
        assert torch.equal(out, ref)


def test_reduce_decode_low_rank_factor():
    d_out, d_in, R = 300, 1024, 4
    F, f = rand_factor(d_out, d_in, seed=53, rank=8)
    gen = torch.Generator(device=DEV).manual_seed(54)
    Ws = [torch.randn(d_out, d_in, generator=gen, device=DEV) for _ in range(R)]
    codes, scales, _ = encode_replicas(f, Ws, "e4m3", "tensor", d_out, d_in)
    avg, _ = two_calls(f, codes, scales, None, "e4m3", "tensor", d_out, d_in)
    out = torch.empty(d_out, d_in, device=DEV)
    G.gift_reduce_decode(ctx(), f, codes, scales, "e4m3", "tensor", d_out, d_in, out,
                         ws=ws("reduce_decode", "lowrank", "e4m3", "tensor", d_out, d_in))
    torch.cuda.synchronize()
    assert rel_fro(out.cpu().numpy(), O.lowrank_unwhiten(avg.cpu().numpy(), F)) <= 1e-5


@pytest.mark.parametrize("case", ["nvfp4", "block128", "identity", "ragged", "chol_input"])
def test_reduce_decode_other_factors_and_formats(case):
    # the same result as the two calls, bit for bit
    d_out, d_in, R = 200, (510 if case == "ragged" else 512), 3
    fmt, scaling = {"nvfp4": ("nvfp4", "tensor"), "block128": ("e5m2", "block128")}.get(case, ("e4m3", "tensor"))
    if case == "identity":
        f = None
    elif case == "chol_input":
        rng = np.random.default_rng(55)
        A = np.cov(rng.standard_normal((d_in, 2 * d_in))) + 0.1 * np.eye(d_in)
        LA = O.cholesky(A).astype(np.float32)
        f = G.Factor("chol_input", d_out, d_in, 32, LA=t(LA), LAinv=t(O.lower_inverse(LA).astype(np.float32)))
    else:
        _, f = rand_factor(d_out, d_in, seed=56)
    gen = torch.Generator(device=DEV).manual_seed(57)
    Ws = [torch.randn(d_out, d_in, generator=gen, device=DEV) for _ in range(R)]
    codes, scales, tsc = encode_replicas(f, Ws, fmt, scaling, d_out, d_in)
    avg, ref = two_calls(f, codes, scales, tsc, fmt, scaling, d_out, d_in)
    kind = "identity" if f is None else f.kind
    avg2 = torch.empty(d_out, d_in, device=DEV)
    out = torch.empty(d_out, d_in, device=DEV)
    st = status()
    G.gift_reduce_decode(ctx(), f, codes, scales, fmt, scaling, d_out, d_in, out, avg_out=avg2, tensor_scales=tsc,
                         ws=ws("reduce_decode", kind, fmt, scaling, d_out, d_in), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(avg2, avg)
    assert torch.equal(out, ref)
