"""GPU parity at the configurations' full sizes:
  - 300M-like fc2: Cholesky factors of A (4096^2, T = 8192 BF16) and G (1024^2) ([notes] core
    idea step 2, eq. (7)), the two-sided and input-only transforms of the 1024 x 4096 gradient
    (eqs. (11), (16)) and their decode (eq. (14));
  - 600M-like fc2: the rank-32 refresh from T = 16384 BF16 activations of 6144 dimensions
    (simplification 2, eq. (17)), checked through the activations (A x = a^T (a x) / T);
  - profiler workload: the heavy-tailed gradients of the two non-square shapes encoded with
    128 x 128 block scales after a rank-32 whitening.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G
from fac_whitening_gb300 import synth

from gpu_util import DEV, ctx, encode, factor_to_gpu, rel_fro, status, t, ws

pytestmark = pytest.mark.gpu


def run_factor(kind, a, d_out, rank=32, delta=None, seed=7, prec="fp32"):
    d_in = a.shape[1]
    f = G.Factor.empty(kind, d_out, d_in, rank)
    n = G.gift_workspace_bytes(ctx(), "factor_update", kind, "e4m3", "tensor", d_out, d_in, a.shape[0], rank)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    G.gift_factor_update(ctx(), f, a, delta=delta, seed=seed, prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    return f, int(st.item())


@pytest.fixture(scope="module")
def c2():
    spec = synth.llama300m_fc2_workload().layers[0]
    Ws, a = synth.layer_inputs(spec, 1, 0, 1)
    delta = synth.delta_for_layer(spec, 1, 0)
    return spec, Ws[0].numpy(), a, delta


def test_c2_cholesky_factors_full_size(c2):
    spec, _, a, delta = c2
    f, st = run_factor("chol_two_sided", a.to(DEV), spec.d_out, delta=delta.to(DEV))
    assert st == 0
    for Lt, Lit, x in ((f.LA, f.LAinv, a), (f.LG, f.LGinv, delta)):
        d = x.shape[1]
        L, Li = Lt.cpu().double().numpy(), Lit.cpu().double().numpy()
        assert np.all(np.triu(L, 1) == 0) and np.all(np.triu(Li, 1) == 0)
        # The factor of the exact A: A is formed on the device by FP32 accumulation over
        # T = 8192 tokens, about sqrt(T) u = 90 x 6e-8 = 5e-6 relative (u the FP32 unit
        # roundoff), and L L^T reproduces it to that.
        A = O.kfac_factor(x.double().numpy())
        assert rel_fro(L @ L.T, A) <= 1e-5
        # The factorisation itself, against the oracle's Cholesky of the device's own A (the
        # same FP32 K-FAC product gift_kfac_factor returns): FP64 on both sides, so the only
        # difference is L and L^-1 rounded to FP32.
        Ag = torch.empty(d, d, device=DEV)
        n = G.gift_workspace_bytes(ctx(), "kfac_factor", "identity", "e4m3", "tensor", d, d, x.shape[0])
        G.gift_kfac_factor(ctx(), x.to(DEV), Ag, prec="fp32", ws=torch.zeros(n, dtype=torch.uint8, device=DEV),
                           status=status())
        torch.cuda.synchronize()
        Lo = O.cholesky(Ag.cpu().double().numpy())
        assert rel_fro(L, Lo) <= 1e-6
        assert rel_fro(Li, O.lower_inverse(Lo)) <= 1e-6


@pytest.mark.parametrize("kind", ["chol_input", "chol_two_sided"])
def test_c2_transform_full_size(c2, kind):
    spec, W, a, delta = c2
    LA = O.cholesky(O.kfac_factor(a.double().numpy()))
    LG = O.cholesky(O.kfac_factor(delta.double().numpy()))
    f32 = lambda x: x.astype(np.float32)   # noqa: E731
    LA, LAi, LG, LGi = f32(LA), f32(O.lower_inverse(LA)), f32(LG), f32(O.lower_inverse(LG))
    f = factor_to_gpu(kind, *W.shape, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    xf = O.Xform(kind, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    out = encode(f, W, "e4m3")
    assert out["status"] == 0
    assert rel_fro(out["tout"], xf.whiten(W)) <= 1e-5
    np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e4m3")["codes"])
    X = np.random.default_rng(8).standard_normal(W.shape).astype(np.float32)
    Wo = torch.empty(*W.shape, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), f, t(X), False, "f32", "tensor", *W.shape, Wo, ws=ws("decode", kind, "f32", "tensor", *W.shape))
    torch.cuda.synchronize()
    assert rel_fro(Wo.cpu().numpy(), xf.unwhiten(X)) <= 1e-5


@pytest.mark.parametrize("prec", ["fp32", "tc"])
def test_c3_lowrank_refresh_full_size(prec):
    spec = synth.llama600m_selective_workload().layers[0]
    _, a = synth.layer_inputs(spec, 2, 0, 1, device="cuda")
    f, st = run_factor("lowrank", a, spec.d_out, prec=prec)
    assert st == 0
    a64 = a.double().cpu().numpy()
    T = a64.shape[0]
    apply_A = lambda X: a64.T @ (a64 @ X) / T   # noqa: E731
    U = f.U.cpu().double().numpy()
    mu = f.mu.cpu().double().numpy()
    np.testing.assert_allclose(U.T @ U, np.eye(32), atol=1e-5)
    # residual bound: some exact eigenvalue of A lies within ||A u - mu u|| of mu
    res = np.linalg.norm(apply_A(U) - U * mu, axis=0)
    assert np.all(res <= 2e-3 * mu), res / mu
    Fo = O.lowrank_factor_from_activations(a64, r=32)
    np.testing.assert_allclose(mu, Fo.mu, rtol=1e-3 if prec == "fp32" else 5e-3)
    tr = float(np.sum(a64 * a64)) / T
    sigma = float(f.sigma.item())
    want = (tr - Fo.mu.sum()) / (spec.d_in - 32)
    assert abs(sigma - want) <= (1e-3 if prec == "fp32" else 5e-3) * want


@pytest.mark.parametrize("prec", ["tc", "fp32"])
def test_c3_kfac_factor_full_size_freivalds(prec):
    # A = a^T a / T at 16384 x 6144 (BF16 activations): 8 seeded probes A x against
    # a^T (a x) / T in FP64, and 4096 sampled entries against their dot products
    spec = synth.llama600m_selective_workload().layers[0]
    _, a = synth.layer_inputs(spec, 2, 0, 1, device="cuda")
    T, d = a.shape
    A = torch.empty(d, d, device=DEV)
    n = G.gift_workspace_bytes(ctx(), "kfac_factor", "identity", "e4m3", "tensor", d, d, T)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    G.gift_kfac_factor(ctx(), a, A, prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    a64 = a.double().cpu().numpy()
    Ah = A.cpu().double().numpy()
    X = np.random.default_rng(21).standard_normal((d, 8))
    assert rel_fro(Ah @ X, a64.T @ (a64 @ X) / T) <= 1e-4
    rng = np.random.default_rng(22)
    i, j = rng.integers(0, d, 4096), rng.integers(0, d, 4096)
    want = np.einsum("ti,ti->i", a64[:, i], a64[:, j]) / T
    assert rel_fro(Ah[i, j], want) <= 1e-4
    np.testing.assert_array_equal(Ah, Ah.T)


def _c4_case(idx, T=16384, exponent=0.8):
    """A profiler-workload gradient (Student-t, per-column log-normal scale) and a rank-32
    factor from T synthetic activations of its input width (the 600M-like scheme)."""
    wl = synth.profiler_workload()
    spec = wl.layers[idx]
    W = synth.layer_inputs(spec, wl.config, idx, 1)[0][0].numpy()
    aspec = synth.LayerSpec("act", spec.d_out, spec.d_in, T=T, exponent=exponent)
    _, a = synth.layer_inputs(aspec, wl.config, 100 + idx, 1, device="cuda")
    F = O.lowrank_factor_from_activations(a.double().cpu().numpy(), r=32)
    F32 = O.LowRankFactor(F.U.astype(np.float32), F.mu.astype(np.float32), np.float32(F.sigma))
    return W, F32


@pytest.mark.parametrize("idx", [1, 2], ids=["1536x6144", "6144x1536"])
def test_c4_block128_lowrank_encode_full_size(idx):
    W, F = _c4_case(idx)
    assert W.shape == ((1536, 6144) if idx == 1 else (6144, 1536))
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    out = encode(f, W, "e4m3", "block128")
    assert out["status"] == 0
    want = O.lowrank_whiten(W, F)
    assert rel_fro(out["tout"], want) <= 1e-5
    q = O.quantize(out["tout"], "e4m3", "block128")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
