"""The two statements of the oracle agree (no GPU).

oracle/gift_oracle.cpp (plain single-threaded C++17, -ffp-contract=off) and
oracle/gift_oracle.py (numpy) are written independently from the same passages and both
answer to every pin in test_oracle_pins.py.  Here they are run on the same seeded inputs of
moderate size: the quantisers, scales, reduce and hit counts must agree bit for bit (they are
FP32 operations written one by one on both sides); the double-precision linear algebra must
agree to rounding (different summation orders); and the OpenMP build of the C++ source must
give exactly the single-threaded build's results.
"""
import numpy as np
import pytest

import oracle.gift_oracle as N

C = pytest.importorskip("oracle.cpp")


def _x(shape, seed, heavy=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape)
    if heavy:
        x = rng.standard_t(3, shape) * np.exp(rng.normal(0, 2, (1, shape[1])))
    return x.astype(np.float32)


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("e5m2", "tensor"), ("e4m3", "block128"),
                                         ("e5m2", "block128"), ("e4m3", "block512"), ("nvfp4", "tensor")])
@pytest.mark.parametrize("heavy", [False, True])
def test_quantisers_bit_identical(fmt, scaling, heavy):
    x = _x((300, 528), 1 + heavy, heavy)
    qn, qc = N.quantize(x, fmt, scaling), C.quantize(x, fmt, scaling)
    np.testing.assert_array_equal(qn["codes"], qc["codes"])
    np.testing.assert_array_equal(np.asarray(qn["scales"]), np.asarray(qc["scales"]))
    if fmt == "nvfp4":
        assert np.float32(qn["tensor_scale"]) == np.float32(qc["tensor_scale"])
    np.testing.assert_array_equal(N.dequantize_any(qn, fmt, scaling), C.dequantize_any(qc, fmt, scaling))
    # a caller amax (the shared scale) as well
    am = np.float32(3.0) if scaling == "tensor" else None
    if am is not None:
        np.testing.assert_array_equal(N.quantize(x, fmt, scaling, am)["codes"], C.quantize(x, fmt, scaling, am)["codes"])


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("nvfp4", "tensor"), ("e5m2", "block128")])
def test_replica_reduce_and_hits_bit_identical(fmt, scaling):
    xs = [_x((130, 272), 10 + r, heavy=True) for r in range(5)]
    qs = [N.quantize(x, fmt, scaling) for x in xs]
    np.testing.assert_array_equal(N.replica_reduce(qs, fmt, scaling), C.replica_reduce(qs, fmt, scaling))
    if fmt != "nvfp4":
        for x in xs:
            assert N.boundary_hits(x, fmt, scaling) == C.boundary_hits(x, fmt, scaling)


def test_linear_algebra_agrees():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((700, 160)) * (np.arange(1, 161) ** -0.8)
    A = N.kfac_factor(a)
    np.testing.assert_allclose(C.kfac_factor(a), A, rtol=1e-12, atol=1e-15)
    L = N.cholesky(A)
    np.testing.assert_allclose(C.cholesky(A), L, rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose(C.lower_inverse(L), N.lower_inverse(L), rtol=1e-8, atol=1e-8)
    W = rng.standard_normal((24, 160))
    np.testing.assert_allclose(C.chol_input_whiten(W, L), N.chol_input_whiten(W, L), rtol=1e-8, atol=1e-8)
    Fn = N.lowrank_factor_from_activations(a, r=32)
    Fc = C.lowrank_factor_from_activations(a, r=32)
    np.testing.assert_allclose(Fc.mu, Fn.mu, rtol=1e-10)
    assert np.isclose(Fc.sigma, Fn.sigma, rtol=1e-10)
    # eigenvectors up to sign: the projectors agree
    np.testing.assert_allclose(Fc.U @ Fc.U.T, Fn.U @ Fn.U.T, atol=1e-8)
    np.testing.assert_allclose(C.lowrank_whiten(W, Fn), N.lowrank_whiten(W, Fn), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(C.lowrank_unwhiten(W, Fn), N.lowrank_unwhiten(W, Fn), rtol=1e-11, atol=1e-12)


def test_encode_layer_with_residual_agrees():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((40, 96))
    R0 = (rng.standard_normal((40, 96)) * 0.01).astype(np.float32)
    qn, tn, rn = N.encode_layer(W, N.Xform("identity"), "e4m3", residual=R0)
    qc, tc, rc = C.encode_layer(W, C.Xform("identity"), "e4m3", residual=R0)
    np.testing.assert_array_equal(tn, tc)
    np.testing.assert_array_equal(qn["codes"], qc["codes"])
    np.testing.assert_array_equal(rn, rc)


def test_openmp_build_is_identical():
    x = _x((512, 1024), 5, heavy=True)
    a = np.random.default_rng(6).standard_normal((400, 200))
    try:
        C.use_openmp(False)
        q1 = C.quantize(x, "nvfp4")
        F1 = C.lowrank_factor_from_activations(a, r=16)
        threads = C.use_openmp(True)
        q2 = C.quantize(x, "nvfp4")
        F2 = C.lowrank_factor_from_activations(a, r=16)
    finally:
        C.use_openmp(False)
    assert threads >= 1
    np.testing.assert_array_equal(q1["codes"], q2["codes"])
    np.testing.assert_array_equal(q1["scales"], q2["scales"])
    np.testing.assert_array_equal(F1.mu, F2.mu)
    np.testing.assert_array_equal(F1.U, F2.U)
