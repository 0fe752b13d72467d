"""GPU factor refresh against the oracle: K-FAC factor (eq. (4)), rank-r eigenpairs
(eq. (17), eigenvalues within 1e-3 relative over the top 32) and the Cholesky
factors (eq. (7): L L^T = A, L^-1 A L^-T = I)."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G
from fac_whitening_gb300 import synth

from gpu_util import DEV, ctx, rel_fro, status, t

pytestmark = pytest.mark.gpu


def run_factor(kind, a, d_out, rank=32, delta=None, seed=7, iters=None, prec="fp32", sketch=0):
    d_in = a.shape[1]
    f = G.Factor.empty(kind, d_out, d_in, rank)
    G.gift_set_option(ctx(), G.OPT_SKETCH, sketch)
    n = G.gift_workspace_bytes(ctx(), "factor_update", kind, "e4m3", "tensor", d_out, d_in, a.shape[0], rank)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    if iters:
        G.gift_set_option(ctx(), G.OPT_SUBSPACE_ITERS, iters)
    G.gift_factor_update(ctx(), f, a, delta=delta, seed=seed, prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    if iters:
        G.gift_set_option(ctx(), G.OPT_SUBSPACE_ITERS, 16)
    G.gift_set_option(ctx(), G.OPT_SKETCH, 0)
    return f, w, int(st.item())


def check_lowrank(f, a64, rank, st, sigma_rtol=1e-3):
    assert st == 0
    A = O.kfac_factor(a64)
    ev = np.sort(np.linalg.eigvalsh(A))[::-1]
    mu = f.mu.cpu().double().numpy()
    U = f.U.cpu().double().numpy()
    np.testing.assert_allclose(mu, ev[:rank], rtol=1e-3)
    d = A.shape[0]
    sigma = float(f.sigma.item())
    want_sigma = 1.0 if rank == d else (np.trace(A) - ev[:rank].sum()) / (d - rank)
    assert abs(sigma - want_sigma) <= sigma_rtol * abs(want_sigma)
    np.testing.assert_allclose(U.T @ U, np.eye(rank), atol=1e-5)
    # residual bound: some exact eigenvalue lies within ||A u - mu u|| of mu
    res = np.linalg.norm(A @ U - U * mu, axis=0)
    assert np.all(res <= 1e-3 * mu), res / mu
    # against the oracle's own factor
    Fo = O.lowrank_factor_from_activations(a64, r=rank)
    np.testing.assert_allclose(mu, Fo.mu, rtol=1e-3)


def test_factor_lowrank_tiny():
    spec = synth.tiny_workload().layers[0]
    _, a = synth.layer_inputs(spec, 0, 0, 1)
    f, w, st = run_factor("lowrank", t(a), 64, sketch=1)   # explicit: A is formed
    check_lowrank(f, a.double().numpy(), 32, st)
    f, _, st = run_factor("lowrank", t(a), 64)              # implicit
    check_lowrank(f, a.double().numpy(), 32, st)
    # the SYRK result sits at the start of the workspace: A = a^T a / T
    A_gpu = w[: 256 * 256 * 4].view(torch.float32).view(256, 256).cpu().double().numpy()
    assert rel_fro(A_gpu, O.kfac_factor(a.double().numpy())) <= 1e-6


@pytest.mark.parametrize("sketch", [0, 1], ids=["implicit", "explicit"])
def test_factor_lowrank_bf16_steep(sketch):
    # the steepest spectrum of the 600M-like layers (exponent 1.2: mu_32 / mu_1 = 2.5e-4); the
    # sketch A Q formed from the activations (a^T (a Q) / T, A never formed) or from A
    spec = synth.LayerSpec("m", 128, 1024, T=4096, exponent=1.2, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 9, 3, 1, device="cuda")
    f, _, st = run_factor("lowrank", a, 128, sketch=sketch)
    check_lowrank(f, a.double().cpu().numpy(), 32, st)


def test_factor_tc_syrk_exact_on_integer_activations():
    # tensor-core SYRK (TC precision, BF16 activations, d % 256 == 0, T % 64 == 0): with small
    # integer activations every partial sum is an exactly representable FP32 integer, so the
    # result must equal a^T a / T exactly (T a power of two), tiles, transpose and mirror included
    rng = np.random.default_rng(11)
    T, d = 1024, 512
    a = rng.integers(-2, 3, size=(T, d)).astype(np.float32)
    at = torch.tensor(a, dtype=torch.bfloat16, device=DEV)
    f, w, st = run_factor("lowrank", at, 256, prec="tc", sketch=1)
    assert st == 0
    A_gpu = w[: d * d * 4].view(torch.float32).view(d, d).cpu().double().numpy()
    np.testing.assert_array_equal(A_gpu, (a.astype(np.float64).T @ a.astype(np.float64)) / T)


def test_factor_lowrank_bf16_steep_tc():
    # same inputs as the FP32 test, A on the tensor cores: eigenvalues within 1e-3, and A
    # itself within the accumulation error of 256 tensor-core K steps.  sigma = (tr A -
    # sum mu) / (d - r) cancels on this steep spectrum (sigma / mu_1 ~ 1e-5), which amplifies
    # the accumulation error; its bound follows from the TC transform tolerance: alpha =
    # sigma^-1/2 moves by half of sigma's relative error, 1e-2 -> 5e-3 < 2e-2
    spec = synth.LayerSpec("m", 128, 1024, T=4096, exponent=1.2, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 9, 3, 1, device="cuda")
    f, w, st = run_factor("lowrank", a, 128, prec="tc", sketch=1)
    a64 = a.double().cpu().numpy()
    check_lowrank(f, a64, 32, st, sigma_rtol=1e-2)
    A_gpu = w[: 1024 * 1024 * 4].view(torch.float32).view(1024, 1024).cpu().double().numpy()
    assert rel_fro(A_gpu, O.kfac_factor(a64)) <= 1e-4


@pytest.mark.parametrize("prec", ["fp32", "tc"])
def test_kfac_factor_entry_point(prec):
    # A = a^T a / T alone, both precisions; integer activations make every sum exact
    rng = np.random.default_rng(13)
    T, d = 512, 256
    a = rng.integers(-3, 4, size=(T, d)).astype(np.float32)
    at = torch.tensor(a, dtype=torch.bfloat16, device=DEV)
    A = torch.empty(d, d, device=DEV)
    n = G.gift_workspace_bytes(ctx(), "kfac_factor", "identity", "e4m3", "tensor", d, d, T)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    G.gift_kfac_factor(ctx(), at, A, prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(A.cpu().double().numpy(), a.astype(np.float64).T @ a.astype(np.float64) / T)


def test_factor_exact_rank_equals_d_in():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal((200, 16)) * np.linspace(2, 0.3, 16)).astype(np.float32)
    f, _, st = run_factor("lowrank", t(a), 8, rank=16)
    check_lowrank(f, a.astype(np.float64), 16, st)
    F = O.LowRankFactor(f.U.cpu().double().numpy(), f.mu.cpu().double().numpy(), f.sigma.item())
    T = O.lowrank_T(F)
    A = O.kfac_factor(a.astype(np.float64))
    np.testing.assert_allclose(T.T @ A @ T, np.eye(16), atol=1e-4)


@pytest.mark.parametrize("kind", ["chol_input", "chol_two_sided"])
def test_factor_cholesky(kind):
    spec = synth.LayerSpec("c", 96, 320, T=2048, exponent=0.5, act_dtype=torch.float32)
    _, a = synth.layer_inputs(spec, 9, 4, 1)
    delta = synth.delta_for_layer(spec, 9, 4)
    f, _, st = run_factor(kind, t(a), 96, delta=t(delta) if kind == "chol_two_sided" else None)
    assert st == 0
    pairs = [(f.LA, f.LAinv, a)]
    if kind == "chol_two_sided":
        pairs.append((f.LG, f.LGinv, delta))
    for Lt, Lit, x in pairs:
        A = O.kfac_factor(x.double().numpy())
        L = Lt.cpu().double().numpy()
        Li = Lit.cpu().double().numpy()
        assert np.all(np.triu(L, 1) == 0) and np.all(np.triu(Li, 1) == 0)
        assert rel_fro(L @ L.T, A) <= 1e-6
        np.testing.assert_allclose(Li @ A @ Li.T, np.eye(A.shape[0]), atol=1e-4)
        assert rel_fro(L, O.cholesky(A)) <= 1e-4


def test_factor_cholesky_not_pd_status():
    a = np.zeros((64, 80), np.float32)           # A = 0: the first pivot is not positive
    f, _, st = run_factor("chol_input", t(a), 8)
    assert st == G.ERR_NOT_PD


def test_philox_start_is_seeded():
    spec = synth.tiny_workload().layers[0]
    _, a = synth.layer_inputs(spec, 0, 1, 1)
    f1, _, _ = run_factor("lowrank", t(a), 64, seed=1)
    f2, _, _ = run_factor("lowrank", t(a), 64, seed=1)
    f3, _, _ = run_factor("lowrank", t(a), 64, seed=2)
    assert torch.equal(f1.U, f2.U) and torch.equal(f1.mu, f2.mu)
    np.testing.assert_allclose(f1.mu.cpu().numpy(), f3.mu.cpu().numpy(), rtol=1e-4)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_factor_fp32_tc_syrk_exact_on_integer_activations(dtype):
    # the FP32-precision K-FAC product on the tensor cores (exact BF16 terms, one accumulator per
    # 64 tokens, round-to-nearest sums): with small integer activations every partial sum is an
    # exact FP32 integer, so A = a^T a / T exactly, ragged row tiles and the mirror included
    rng = np.random.default_rng(12)
    T, d = 1024, 320
    a = rng.integers(-3, 4, size=(T, d)).astype(np.float32)
    at = torch.tensor(a, dtype=dtype, device=DEV)
    A = torch.empty(d, d, device=DEV)
    n = G.gift_workspace_bytes(ctx(), "kfac_factor", "identity", "e4m3", "tensor", d, d, T)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    G.gift_kfac_factor(ctx(), at, A, prec="fp32", ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(A.cpu().double().numpy(), (a.astype(np.float64).T @ a.astype(np.float64)) / T)


def test_refresh_iterations_stop_when_ritz_values_settle():
    # the convergence stop: a cap of 40 iterations gives the same factor as a cap of 12 once the
    # Ritz values have settled (the remaining iterations do nothing)
    spec = synth.LayerSpec("m", 128, 1024, T=4096, exponent=0.8, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 9, 4, 1, device="cuda")
    f12, _, st12 = run_factor("lowrank", a, 128, iters=12)
    f40, _, st40 = run_factor("lowrank", a, 128, iters=40)
    assert st12 == 0 and st40 == 0
    assert torch.equal(f12.mu, f40.mu) and torch.equal(f12.U, f40.U)
    check_lowrank(f40, a.double().cpu().numpy(), 32, st40)


def kfac_on_gpu(a, prec="fp32"):
    T, d = a.shape
    A = torch.empty(d, d, device=DEV)
    n = G.gift_workspace_bytes(ctx(), "kfac_factor", "identity", "e4m3", "tensor", d, d, T)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    G.gift_kfac_factor(ctx(), a, A, prec=prec, ws=w)
    return A


def from_kfac(kind, A, d_out, Gm=None, rank=32, seed=7):
    d_in = A.shape[0]
    f = G.Factor.empty(kind, d_out, d_in, rank)
    n = G.gift_workspace_bytes(ctx(), "factor_update", kind, "e4m3", "tensor", d_out, d_in, 0, rank)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    G.gift_factor_update_from_kfac(ctx(), f, A, Gm, seed=seed, ws=w, status=st)
    torch.cuda.synchronize()
    return f, int(st.item())


@pytest.mark.parametrize("d_in", [1024, 64], ids=["tensor-core", "small"])
def test_from_kfac_replica_average(d_in):
    # the factor of A averaged over four replicas' K-FAC factors equals the factor of all their
    # activations together (equal T per replica): eigenpairs checked against the concatenation
    spec = synth.LayerSpec("m", 128, d_in, T=1024, exponent=1.2, act_dtype=torch.bfloat16)
    Q = synth.haar_orthogonal(d_in, synth.seed_for(9, 3, stream=1), device="cuda")
    s = synth.layer_spectrum(spec, 9, 3, device="cuda")
    acts = [synth.activations(spec.T, d_in, s, Q, synth.seed_for(9, 3, r, stream=2), "cuda", torch.bfloat16)
            for r in range(4)]
    A = sum(kfac_on_gpu(a) for a in acts) / 4.0
    f, st = from_kfac("lowrank", A, 128)
    a64 = torch.cat(acts).double().cpu().numpy()
    check_lowrank(f, a64, 32, st)


def test_from_kfac_matches_activations_path():
    # the explicit-sketch refresh from the activations and the refresh from the same A agree
    # within the eigenvalue tolerance (they differ only in how the last Rayleigh-Ritz step forms
    # Q^T A Q), with the trace and so sigma taken from the same A
    spec = synth.LayerSpec("m", 128, 2048, T=2048, exponent=1.0, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 5, 1, 1, device="cuda")
    f1, _, st1 = run_factor("lowrank", a, 128, sketch=1)
    f2, st2 = from_kfac("lowrank", kfac_on_gpu(a), 128)
    assert st1 == 0 and st2 == 0
    np.testing.assert_allclose(f2.mu.cpu().numpy(), f1.mu.cpu().numpy(), rtol=1e-3)
    assert abs(float(f2.sigma.item()) - float(f1.sigma.item())) <= 1e-3 * abs(float(f1.sigma.item()))
    check_lowrank(f2, a.double().cpu().numpy(), 32, st2)


@pytest.mark.parametrize("kind", ["chol_input", "chol_two_sided"])
def test_from_kfac_cholesky_bit_identical(kind):
    # the Cholesky kinds from A (and G) formed by gift_kfac_factor give the same factors, bit
    # for bit, as the refresh from the activations (the same K-FAC product, the same FP64 factoring)
    rng = np.random.default_rng(21)
    T, d_in, d_out = 1024, 384, 256
    a = t(rng.standard_normal((T, d_in)))
    delta = t(rng.standard_normal((T, d_out))) if kind == "chol_two_sided" else None
    f1, _, st1 = run_factor(kind, a, d_out, delta=delta)
    A = kfac_on_gpu(a)
    Gm = kfac_on_gpu(delta) if delta is not None else None
    f2, st2 = from_kfac(kind, A, d_out, Gm=Gm)
    assert st1 == 0 and st2 == 0
    assert torch.equal(f1.LA, f2.LA) and torch.equal(f1.LAinv, f2.LAinv)
    if kind == "chol_two_sided":
        assert torch.equal(f1.LG, f2.LG) and torch.equal(f1.LGinv, f2.LGinv)
    # and L L^T = A for the given A
    LA = f2.LA.cpu().double().numpy()
    assert rel_fro(LA @ LA.T, A.cpu().double().numpy()) <= 1e-5


def test_refresh_replays_from_a_cuda_graph():
    # the rank-r refresh is a fixed launch sequence that allocates nothing and never waits on
    # the host (its convergence test only makes later launches return at once): captured
    # once into a CUDA graph, a replay gives the eager call's factor bit for bit
    spec = synth.LayerSpec("g", 128, 1024, T=4096, exponent=1.2, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 9, 3, 1, device="cuda")
    n = G.gift_workspace_bytes(ctx(), "factor_update", "lowrank", "e4m3", "tensor", 128, 1024, a.shape[0], 32)
    w = torch.zeros(n, dtype=torch.uint8, device=DEV)
    st = status()
    eager = G.Factor.empty("lowrank", 128, 1024, 32)
    G.gift_factor_update(ctx(), eager, a, seed=7, ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    f = G.Factor.empty("lowrank", 128, 1024, 32)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        G.gift_factor_update(ctx(), f, a, seed=7, ws=w, status=st)
    g.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in ((f.U, eager.U), (f.mu, eager.mu), (f.sigma, eager.sigma)):
        assert torch.equal(x, y)
    check_lowrank(f, a.double().cpu().numpy(), 32, 0)
