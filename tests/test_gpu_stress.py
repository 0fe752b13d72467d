"""GPU parity at the large-stress size: fc2-like layers of 4096 x 16384, rank 32, NVFP4 and
E4M3 side by side, R = 16 replica buffers dequantised and averaged in HBM.

The factor is a synthetic rank-32 one: U is orthonormal, and mu is the spectrum i^-1 with
8 of its entries raised 100x.  No activations are used, since the factor update at this
size is a separate test.  The checks use the same contracts as the smaller parity tests:
- the transform on the whole tensor, within 1e-5 of the oracle's;
- the quantiser contract, bit-exact on sampled rows (the per-tensor scale comes from the
  whole tensor's amax);
- the 16-replica reduce, bit-exact on sampled rows (every row is independent);
- the decode of the reduced tensor on the whole tensor, within 1e-5."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G

from gpu_util import DEV, alloc_codes, ctx, rel_fro, status, t, ws

pytestmark = pytest.mark.gpu
D_OUT, D_IN, R = 4096, 16384, 16
TOL = 1e-5
ROWS = np.array([0, 1, 127, 128, 2047, 2048, 4094, 4095])


@pytest.fixture(scope="module")
def layer():
    rng = np.random.default_rng(61)
    U, _ = np.linalg.qr(rng.standard_normal((D_IN, 32)))
    spec = 1.0 / np.arange(1, 33)
    spec[rng.choice(32, 8, replace=False)] *= 100.0
    mu = np.sort(spec)[::-1].copy()
    F = O.LowRankFactor(U.astype(np.float32), mu.astype(np.float32), np.float32(0.01))
    f = G.Factor("lowrank", D_OUT, D_IN, 32, U=t(F.U), mu=t(F.mu), sigma=t([F.sigma]))
    gen = torch.Generator(device=DEV).manual_seed(62)
    Ws = []
    for _ in range(R):
        W = torch.randn(D_OUT, D_IN, generator=gen, device=DEV) * 0.1
        W += (torch.randn(D_OUT, 32, generator=gen, device=DEV) * 3.0) @ f.U.T
        Ws.append(W.contiguous())
    return F, f, Ws


def quantize_rows(x_rows, amax, fmt):
    return O.quantize(x_rows, fmt, "tensor", amax=amax)


@pytest.mark.parametrize("fmt", ["e4m3", "nvfp4"])
def test_stress_encode(layer, fmt):
    F, f, Ws = layer
    codes, scales, tscale = alloc_codes(fmt, "tensor", D_OUT, D_IN)
    tout = torch.empty(D_OUT, D_IN, dtype=torch.float32, device=DEV)
    st = status()
    G.gift_encode(ctx(), f, Ws[0], fmt, "tensor", codes, scales, tscale, transformed_out=tout,
                  ws=ws("encode", "lowrank", fmt, "tensor", D_OUT, D_IN), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    X = tout.cpu().numpy()
    assert rel_fro(X, O.lowrank_whiten(Ws[0].cpu().numpy(), F)) <= TOL
    amax = O.abs_max(X)
    q = quantize_rows(X[ROWS], amax, fmt)
    if fmt == "nvfp4":
        np.testing.assert_array_equal(codes.view(D_OUT, D_IN // 2).cpu().numpy()[ROWS], q["codes"])
        np.testing.assert_array_equal(scales.view(D_OUT, D_IN // 16).cpu().numpy()[ROWS], q["scales"])
        assert tscale.item() == q["tensor_scale"]
    else:
        np.testing.assert_array_equal(codes.view(D_OUT, D_IN).cpu().numpy()[ROWS], q["codes"])
        assert scales.item() == q["scales"][0]


@pytest.mark.parametrize("fmt", ["e4m3", "nvfp4"])
def test_stress_replicas_reduce_decode(layer, fmt):
    F, f, Ws = layer
    outs = [alloc_codes(fmt, "tensor", D_OUT, D_IN) for _ in range(R)]
    st = status()
    G.gift_encode_replicas(ctx(), f, Ws, fmt, "tensor", [o[0] for o in outs], scales=[o[1] for o in outs],
                           tensor_scales=[o[2] for o in outs] if fmt == "nvfp4" else None,
                           ws=ws("encode", "lowrank", fmt, "tensor", D_OUT, D_IN), status=st)
    avg = torch.empty(D_OUT, D_IN, dtype=torch.float32, device=DEV)
    G.gift_replica_reduce(ctx(), [o[0] for o in outs], [o[1] for o in outs], fmt, "tensor", D_OUT, D_IN, avg,
                          tensor_scales=[o[2] for o in outs] if fmt == "nvfp4" else None, status=st)
    Wo = torch.empty(D_OUT, D_IN, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), f, avg, False, "f32", "tensor", D_OUT, D_IN, Wo,
                  ws=ws("decode", "lowrank", "f32", "tensor", D_OUT, D_IN), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the reduce, row by row: each replica dequantised with its own scales, added in order
    qs = []
    for c, s, ts in outs:
        if fmt == "nvfp4":
            qs.append({"codes": c.view(D_OUT, D_IN // 2).cpu().numpy()[ROWS],
                       "scales": s.view(D_OUT, D_IN // 16).cpu().numpy()[ROWS], "tensor_scale": np.float32(ts.item())})
        else:
            qs.append({"codes": c.view(D_OUT, D_IN).cpu().numpy()[ROWS], "scales": s.cpu().numpy(),
                       "tensor_scale": None})
    np.testing.assert_array_equal(avg.cpu().numpy()[ROWS], O.replica_reduce(qs, fmt))
    # the decode of the reduced tensor, whole
    assert rel_fro(Wo.cpu().numpy(), O.lowrank_unwhiten(avg.cpu().numpy(), F)) <= TOL
