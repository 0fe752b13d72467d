"""Pins of the CPU oracle to things outside itself (no GPU).

Each test checks an oracle function against what the GIFT pages print, a closed
form, an invariant, a library routine, or brute force on a tiny input, chosen so
that a dropped term, a wrong sign or index, or a transposed operand fails.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.gift_oracle as oracle_numpy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# Both statements of the oracle (numpy, and the single-threaded C++ library) answer to every pin.
@pytest.fixture(params=["numpy", "cpp"], scope="module")
def O(request):
    if request.param == "numpy":
        return oracle_numpy
    import oracle.cpp as oracle_cpp
    return oracle_cpp


# ---------------------------------------------------------------------------------------
# helpers independent of the oracle
# ---------------------------------------------------------------------------------------

def brute_values(ebits, mbits, bias):
    """All finite non-negative values of a minifloat by enumerating its bit fields."""
    vals = {}
    for e in range(1 << ebits):
        for m in range(1 << mbits):
            if e == 0:
                v = m * 2.0 ** (1 - bias - mbits)
            else:
                v = (1 + m / 2 ** mbits) * 2.0 ** (e - bias)
            vals[(e << mbits) | m] = v
    return vals


def brute_encode(y, fmt_fields, maxval, nbits):
    """Nearest representable value by exhaustive search; ties to the even code."""
    ebits, mbits, bias = fmt_fields
    table = {c: v for c, v in brute_values(ebits, mbits, bias).items() if v <= maxval}
    out = []
    for yy in np.asarray(y, dtype=np.float32).astype(np.float64):
        a = abs(yy)
        if a >= maxval:
            best = max(table, key=lambda c: table[c])
        else:
            dmin = min(abs(v - a) for v in table.values())
            cands = [c for c, v in table.items() if abs(v - a) == dmin]
            if len(cands) > 1:
                cands = [c for c in cands if c % 2 == 0]
            best = cands[0]
        sign = 1 if math.copysign(1.0, yy) < 0 else 0
        out.append((sign << (nbits - 1)) | best)
    return np.array(out, dtype=np.uint8)


def probe_values(fmt_fields, maxval):
    """Midpoints between adjacent values, one FP32 ulp either side, beyond max, random."""
    vals = sorted(set(v for v in brute_values(*fmt_fields).values() if v <= maxval))
    pts = []
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = np.float32((lo + hi) / 2)
        pts += [lo, hi, mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))]
    pts += [maxval * 1.01, maxval * 1.0625, maxval * 2, 3.4e38, 1e-30, 1e-45, 0.0]
    rng = np.random.default_rng(7)
    pts += list(rng.uniform(0, maxval * 1.1, 500)) + list(np.exp(rng.uniform(-25, np.log(maxval), 500)))
    p = np.array(pts, dtype=np.float32)
    return np.concatenate([p, -p])


FIELDS = {"e4m3": ((4, 3, 7), 448.0, 8), "e5m2": ((5, 2, 15), 57344.0, 8), "e2m1": ((2, 1, 1), 6.0, 4)}
def OFMT(O):
    return {"e4m3": O.E4M3, "e5m2": O.E5M2, "e2m1": O.E2M1}


# ---------------------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------------------

def test_format_constants_from_pages(O):
    # GIFT reading notes, prerequisites, "What FP8 is": E4M3 max ~448, E5M2 max ~57344,
    # 2^3 or 2^2 mantissa levels per octave.
    assert O.decode([O.E4M3.max_code], O.E4M3)[0] == 448.0
    assert O.decode([O.E5M2.max_code], O.E5M2)[0] == 57344.0
    assert O.E4M3.max_code == 0x7E and O.E5M2.max_code == 0x7B
    for fmt, levels in ((O.E4M3, 8), (O.E5M2, 4)):
        codes = np.arange(128)
        v = O.decode(codes, fmt)
        assert np.count_nonzero((v >= 1.0) & (v < 2.0)) == levels
        assert np.count_nonzero((v >= 64.0) & (v < 128.0)) == levels
    assert O.decode([1], O.E4M3)[0] == 2.0 ** -9
    assert O.decode([1], O.E5M2)[0] == 2.0 ** -16
    assert list(O.decode(np.arange(8), O.E2M1)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert np.isnan(O.decode([0x7F], O.E4M3)[0]) and np.isinf(O.decode([0x7C], O.E5M2)[0])


@pytest.mark.parametrize("name,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_decode_matches_torch_float8(O, name, tdt):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(tdt).to(torch.float64).numpy()
    got = O.decode(codes, OFMT(O)[name])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("name", ["e4m3", "e5m2", "e2m1"])
def test_encode_matches_brute_force(O, name):
    fields, maxval, nbits = FIELDS[name]
    y = probe_values(fields, maxval)
    np.testing.assert_array_equal(O.encode(y, OFMT(O)[name]), brute_encode(y, fields, maxval, nbits))


@pytest.mark.parametrize("name,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_encode_matches_torch_in_range(O, name, tdt):
    fields, maxval, _ = FIELDS[name]
    y = probe_values(fields, maxval)
    y = y[np.abs(y) < maxval]
    ref = torch.from_numpy(y).to(tdt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.encode(y, OFMT(O)[name]), ref)


# ---------------------------------------------------------------------------------------
# scaling + quantisation
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["e4m3", "e5m2"])
def test_quantize_8x8_brute_force(O, name):
    # the scale rule s = amax/FP8_MAX (prerequisites, "What FP8 is"); codes by exhaustive search
    fields, maxval, nbits = FIELDS[name]
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((8, 8)) * np.exp(rng.uniform(-6, 3, (8, 8)))).astype(np.float32)
    codes, s, amax = O.quantize_tensor(x, OFMT(O)[name])
    assert amax == np.max(np.abs(x))
    assert s == np.float32(amax) / np.float32(maxval)
    m = np.float32(maxval) / np.float32(amax)
    y = (x * m).astype(np.float32)
    np.testing.assert_array_equal(codes, brute_encode(y.ravel(), fields, maxval, nbits).reshape(8, 8))
    # the largest element lands on the format's largest value
    assert (int(codes.ravel()[np.argmax(np.abs(x))]) & 0x7F) == OFMT(O)[name].max_code


def test_dequant_error_bound(O):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(4096).astype(np.float32) * 3
    codes, s, _ = O.quantize_tensor(x, O.E4M3)
    xh = O.dequantize(codes, s, O.E4M3).astype(np.float64)
    # half a unit of the 3-bit mantissa (2^-4 relative) in the normal range, half a
    # subnormal step (2^-10 * s) below it, plus rounding of the scale
    bound = np.abs(x) * 2.0 ** -4 * 1.001 + float(s) * 2.0 ** -10 * 1.001
    assert np.all(np.abs(xh - x) <= bound)


def test_zero_and_tiny_amax(O):
    codes, s, amax = O.quantize_tensor(np.array([0.0, -0.0, 0.0], np.float32), O.E4M3)
    assert s == 0 and amax == 0 and list(codes) == [0, 0x80, 0]
    x = np.array([1e-40, -1e-40, 0.0], np.float32)   # subnormal amax: m overflows, clamped
    codes, s, _ = O.quantize_tensor(x, O.E4M3)
    assert np.all(np.isfinite(O.decode(codes, O.E4M3)))


def test_nonfinite_raises(O):
    with pytest.raises(O.NonFinite):
        O.quantize_tensor(np.array([1.0, np.nan], np.float32), O.E4M3)
    with pytest.raises(O.NonFinite):
        O.quantize_tensor(np.array([1.0, np.inf], np.float32), O.E5M2)


def test_block128_tiles_and_edges(O):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((300, 200)).astype(np.float32)
    x[130:140, 150:160] *= 100
    codes, scales, am = O.quantize_block128(x, O.E4M3)
    assert scales.shape == (3, 2)
    for i in range(3):
        for j in range(2):
            t = x[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert am[i, j] == np.max(np.abs(t))
            c, s, _ = O.quantize_tensor(t, O.E4M3)
            np.testing.assert_array_equal(codes[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128], c)
            assert scales[i, j] == s


def test_nvfp4_brute_force(O):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((5, 64)) * np.exp(rng.uniform(-4, 4, (5, 1)))).astype(np.float32)
    packed, bs, st, at = O.quantize_nvfp4(x)
    assert at == np.max(np.abs(x))
    assert st == np.float32(at) / np.float32(2688.0)
    assert packed.shape == (5, 32) and bs.shape == (5, 4)
    f4, _, _ = FIELDS["e2m1"]
    for r in range(5):
        for b in range(4):
            g = x[r, b * 16:(b + 1) * 16]
            ratio = np.float32(np.max(np.abs(g))) / np.float32(np.float32(6.0) * st)
            assert bs[r, b] == brute_encode([ratio], (4, 3, 7), 448.0, 8)[0]
            eb = O.decode([bs[r, b]], O.E4M3)[0]
            eff = np.float32(np.float32(eb) * st)
            rb = np.float32(1.0) / eff
            y = (g * rb).astype(np.float32)
            codes = brute_encode(y, f4, 6.0, 4)
            lo = packed[r, b * 8:(b + 1) * 8] & 0xF
            hi = packed[r, b * 8:(b + 1) * 8] >> 4
            np.testing.assert_array_equal(lo, codes[0::2])
            np.testing.assert_array_equal(hi, codes[1::2])
    xh = O.dequantize_nvfp4(packed, bs, st)
    # value(code) * value(e_b) is exact in FP32 (<= 2 + 4 significant bits)
    c = np.zeros((5, 64), np.uint8)
    c[:, 0::2], c[:, 1::2] = packed & 0xF, packed >> 4
    prod64 = O.decode(c, O.E2M1).reshape(5, 4, 16) * O.decode(bs, O.E4M3)[:, :, None]
    assert np.all(prod64.astype(np.float32).astype(np.float64) == prod64)
    assert np.max(np.abs(xh - x)) <= np.max(np.abs(x)) * 0.5


# ---------------------------------------------------------------------------------------
# replica reduce (eq. (1): g_bar = (1/R) sum_r g^(r))
# ---------------------------------------------------------------------------------------

def test_replica_reduce_exact_mean(O):
    # codes and power-of-two scales chosen so that every partial sum is exact: the
    # result must then equal the mathematical mean of eq. (1)
    rng = np.random.default_rng(8)
    R, n = 8, 257
    qs, exact = [], [Fraction(0)] * n
    for r in range(R):
        vals = rng.integers(-16, 17, n).astype(np.float32)     # exact in E4M3
        s = np.float32(2.0 ** -int(rng.integers(0, 4)))
        codes = O.encode(vals, O.E4M3)
        qs.append({"codes": codes, "scales": np.array([s], np.float32), "tensor_scale": None})
        exact = [e + Fraction(float(v)) * Fraction(float(s)) for e, v in zip(exact, vals)]
    out = O.replica_reduce(qs, "e4m3")
    np.testing.assert_array_equal(out, np.array([float(e / R) for e in exact], np.float32))


def test_replica_reduce_single_is_dequant(O):
    x = np.random.default_rng(9).standard_normal((7, 33)).astype(np.float32)
    q = O.quantize(x, "e5m2")
    np.testing.assert_array_equal(O.replica_reduce([q], "e5m2"), O.dequantize_any(q, "e5m2"))


# ---------------------------------------------------------------------------------------
# boundary-hit profiler (three simplifications, simplification 3)
# ---------------------------------------------------------------------------------------

def test_boundary_hits_hand_example(O):
    # amax = 1 -> m = 448: 1 -> 448 (upper), -1 -> -448 (upper), 0.5 -> 224,
    # 1e-6 -> 4.48e-4 < 2^-10 flushes to zero (lower), 0 is not counted, 3e-4 -> 0.1344
    x = np.array([1.0, -1.0, 0.5, 1e-6, 0.0, 3e-4], np.float32)
    assert O.boundary_hits(x, "e4m3") == (2, 1, 6)
    # E5M2: m = 57344: 1e-6 -> 0.057 is representable (subnormal step 2^-16)
    assert O.boundary_hits(x, "e5m2") == (2, 0, 6)


def test_boundary_hits_brute_force(O):
    rng = np.random.default_rng(10)
    x = (rng.standard_t(3, (40, 50)) * np.exp(2 * rng.standard_normal(50))).astype(np.float32)
    x[0, :5] = 0
    for name in ("e4m3", "e5m2"):
        fields, maxval, nbits = FIELDS[name]
        amax = np.max(np.abs(x))
        m = np.float32(maxval) / np.float32(amax)
        codes = brute_encode((x * m).astype(np.float32).ravel(), fields, maxval, nbits)
        vals = np.abs(O.decode(codes, OFMT(O)[name]))
        up = sum(1 for v in vals if v == maxval)
        lo = sum(1 for v, xx in zip(vals, x.ravel()) if v == 0 and xx != 0)
        assert O.boundary_hits(x, name) == (up, lo, x.size)


def test_block1d_single_block_is_per_tensor(O):
    x = np.random.default_rng(40).standard_normal((20, 25)).astype(np.float32)   # 500 elements
    for name in ("e4m3", "e5m2"):
        c, s, a = O.quantize_block1d(x, OFMT(O)[name])
        ct, st, at = O.quantize_tensor(x, OFMT(O)[name])
        np.testing.assert_array_equal(c, ct)
        assert s.shape == (1,) and s[0] == st and a[0] == at


def test_block1d_power_of_two_copies(O):
    # blocks that are power-of-two multiples of one block: identical codes, scales in the
    # same ratios exactly; a block boundary off by any amount mixes scales and breaks this
    base = np.random.default_rng(41).standard_normal(512).astype(np.float32)
    ks = [-3, 0, 2, 5]
    x = np.stack([base * np.float32(2.0 ** k) for k in ks]).reshape(8, 256)
    for name in ("e4m3", "e5m2"):
        c, s, _ = O.quantize_block1d(x, OFMT(O)[name])
        blocks = c.reshape(4, 512)
        for i in range(4):
            np.testing.assert_array_equal(blocks[i], blocks[1])
            assert s[i] == s[1] * np.float32(2.0 ** ks[i])


def test_block1d_ragged_tail_and_roundtrip(O):
    rng = np.random.default_rng(42)
    x = rng.standard_normal((10, 100)).astype(np.float32)      # 1000 elements: 512 + 488
    x.ravel()[900] = 1000.0                                     # an outlier in the short block
    q = O.quantize(x, "e4m3", "block512")
    assert q["scales"].shape == (2,)
    ct, st, _ = O.quantize_tensor(x.ravel()[:512], OFMT(O)["e4m3"])
    np.testing.assert_array_equal(q["codes"].ravel()[:512], ct)
    assert q["scales"][0] == st and q["scales"][1] == np.float32(1000.0) / np.float32(448.0)
    # round trip within half a code step of the scaled value, plus the subnormal step
    xh = O.dequantize_any(q, "e4m3", "block512")
    s_el = np.repeat(q["scales"], 512)[:1000].reshape(x.shape).astype(np.float64)
    bound = np.abs(x) * 2.0 ** -4 + O.FORMATS["e4m3"].min_subnormal * s_el
    assert np.all(np.abs(xh.astype(np.float64) - x) <= bound * 1.0001)


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("e5m2", "tensor"), ("e4m3", "block128"),
                                         ("e5m2", "block512"), ("nvfp4", "tensor")])
def test_quantisers_are_power_of_two_equivariant(O, fmt, scaling):
    # scaling a tensor by 2^k scales amax, s and every block amax by 2^k exactly and leaves
    # every scaled value x * m unchanged: the codes must not move and the stored scales must
    # scale exactly (the NVFP4 block scales are ratios of amaxes and must not move either)
    x = np.random.default_rng(43).standard_normal((200, 320)).astype(np.float32)
    x[3, :7] = 0
    q0 = O.quantize(x, fmt, scaling)
    for k in (-20, -3, 5, 30):
        qk = O.quantize(x * np.float32(2.0 ** k), fmt, scaling)
        np.testing.assert_array_equal(qk["codes"], q0["codes"])
        if fmt == "nvfp4":
            np.testing.assert_array_equal(qk["scales"], q0["scales"])
            assert qk["tensor_scale"] == q0["tensor_scale"] * np.float32(2.0 ** k)
        else:
            np.testing.assert_array_equal(qk["scales"], q0["scales"] * np.float32(2.0 ** k))


def test_transforms_are_homogeneous_in_the_factor(O):
    # A -> c A: T_A -> c^-1/2 T_A (whitening scales by c^-1/2, map-back by c^1/2), for the
    # sigma-completed rank-r factor and for the Cholesky factor (L -> c^1/2 L)
    rng = np.random.default_rng(44)
    W = rng.standard_normal((6, 40))
    X = rng.standard_normal((6, 40))
    A = _spd(40, 7)
    F = O.lowrank_factor_from_A(A, r=8)
    c = 9.0
    Fc = O.LowRankFactor(F.U, F.mu * c, F.sigma * c)
    np.testing.assert_allclose(O.lowrank_whiten(W, Fc), O.lowrank_whiten(W, F) / 3.0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(O.lowrank_unwhiten(X, Fc), O.lowrank_unwhiten(X, F) * 3.0, rtol=1e-12, atol=1e-14)
    L = O.cholesky(A)
    np.testing.assert_allclose(O.cholesky(c * A), 3.0 * L, rtol=1e-12, atol=1e-14)
    xf, xfc = O.Xform("chol_input", LA=L), O.Xform("chol_input", LA=3.0 * L)
    np.testing.assert_allclose(xfc.whiten(W), xf.whiten(W) / 3.0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(xfc.unwhiten(X), xf.unwhiten(X) * 3.0, rtol=1e-12, atol=1e-14)


def test_select_fragile_ties(O):
    assert O.select_fragile([0.1, 0.3, 0.3, 0.05, 0.2], 3) == [1, 2, 4]


# ---------------------------------------------------------------------------------------
# factors, Cholesky, whitening identities (core idea, eqs. (4)-(14))
# ---------------------------------------------------------------------------------------

def _spd(n, seed, cond=1e3):
    from fac_whitening_gb300 import synth
    return synth.spd_matrix(n, cond, seed).numpy()


def test_kfac_factor_matches_outer_products(O):
    a = np.random.default_rng(11).standard_normal((9, 4))
    A = sum(np.outer(r, r) for r in a) / 9
    np.testing.assert_allclose(O.kfac_factor(a), A, rtol=1e-14, atol=1e-15)


def test_global_factor_is_the_stacked_factor(O):
    # the replica-averaged factor (1/R) sum_r a_r^T a_r / T, for replicas of equal T, is the
    # factor of the replicas' activations stacked into one batch of R T rows
    rng = np.random.default_rng(12)
    acts = [rng.standard_normal((16, 5)) * (1 + r) for r in range(4)]
    mean = sum(O.kfac_factor(x) for x in acts) / len(acts)
    np.testing.assert_allclose(O.kfac_factor(np.concatenate(acts)), mean, rtol=1e-13, atol=1e-14)


def test_cholesky_vs_lapack_and_identities(O):
    A = _spd(24, 1)
    L = O.cholesky(A)
    np.testing.assert_allclose(L, np.linalg.cholesky(A), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(L @ L.T, A, atol=1e-12)
    Li = O.lower_inverse(L)
    np.testing.assert_allclose(Li @ L, np.eye(24), atol=1e-10)
    np.testing.assert_allclose(Li @ A @ Li.T, np.eye(24), atol=1e-10)
    with pytest.raises(O.NotPositiveDefinite):
        O.cholesky(np.array([[1.0, 2.0], [2.0, 1.0]]))


def test_triangular_solves_vs_scipy(O):
    import scipy.linalg as sl
    rng = np.random.default_rng(12)
    LA = O.cholesky(_spd(10, 2))
    LG = O.cholesky(_spd(6, 3))
    W = rng.standard_normal((6, 10))
    # X L_A^T = W  <=>  L_A X^T = W^T
    X = sl.solve_triangular(LA, W.T, lower=True).T
    np.testing.assert_allclose(O.solve_right_lower_t(W, LA), X, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(O.solve_left_lower(LG, W), sl.solve_triangular(LG, W, lower=True),
                               rtol=1e-10, atol=1e-12)


def test_eq9_kfac_norm_equals_whitened_frobenius(O):
    # ||dW||^2_F_W = vec(dW)^T (A (x) G) vec(dW) = ||L_G^T dW L_A||_F^2 (eqs. (5), (9)), vec = column stacking
    rng = np.random.default_rng(13)
    A, G = _spd(4, 4, 50), _spd(3, 5, 20)
    dW = rng.standard_normal((3, 4))
    v = dW.ravel(order="F")
    lhs = v @ np.kron(A, G) @ v
    assert np.isclose(lhs, np.trace(A @ dW.T @ G @ dW), rtol=1e-12)
    LA, LG = O.cholesky(A), O.cholesky(G)
    assert np.isclose(lhs, np.sum((LG.T @ dW @ LA) ** 2), rtol=1e-12)


def test_eq12_two_sided_transform_kronecker_form(O):
    # vec(W~) = (L_A^-1 (x) L_G^-1) vec(W_g)  (eq. (12)); catches transposed or swapped factors
    rng = np.random.default_rng(14)
    A, G = _spd(5, 6, 30), _spd(4, 7, 30)
    LA, LG = O.cholesky(A), O.cholesky(G)
    W = rng.standard_normal((4, 5))
    K = np.kron(np.linalg.inv(LA), np.linalg.inv(LG))
    np.testing.assert_allclose(O.chol_two_sided_whiten(W, LG, LA).ravel(order="F"), K @ W.ravel(order="F"),
                               rtol=1e-10, atol=1e-12)
    # the whitened Fisher is the identity: (L_A^-1 (x) L_G^-1)(A (x) G)(...)^T = I
    np.testing.assert_allclose(K @ np.kron(A, G) @ K.T, np.eye(20), atol=1e-9)
    # input side only (eq. (16) with T_A = L_A^-T) is the same with G = I
    Ki = np.kron(np.linalg.inv(LA), np.eye(4))
    np.testing.assert_allclose(O.chol_input_whiten(W, LA).ravel(order="F"), Ki @ W.ravel(order="F"),
                               rtol=1e-10, atol=1e-12)


def test_whitening_with_given_inverses_matches_solves(O):
    # eq. (11) written with L^-1 (factor carries the inverses) equals the triangular solves
    rng = np.random.default_rng(26)
    LA, LG = O.cholesky(_spd(30, 27, 1e4)), O.cholesky(_spd(7, 28, 1e2))
    W = rng.standard_normal((7, 30))
    np.testing.assert_allclose(O.chol_whiten_with_inverses(W, O.lower_inverse(LA)), O.chol_input_whiten(W, LA),
                               rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(O.chol_whiten_with_inverses(W, O.lower_inverse(LA), O.lower_inverse(LG)),
                               O.chol_two_sided_whiten(W, LG, LA), rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("kind", ["identity", "lowrank", "chol_input", "chol_two_sided"])
def test_eq14_map_back_inverts_eq11(O, kind):
    # with a lossless format the map back is exact (common confusions: lossless GIFT = baseline)
    rng = np.random.default_rng(15)
    d_out, d_in = 6, 40
    A = _spd(d_in, 16, 1e4)
    G = _spd(d_out, 17, 1e2)
    F = O.lowrank_factor_from_A(A, r=8)
    xf = O.Xform(kind, F=F, LA=O.cholesky(A), LG=O.cholesky(G))
    W = rng.standard_normal((d_out, d_in))
    np.testing.assert_allclose(xf.unwhiten(xf.whiten(W)), W, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------------------------------
# low-rank factor (simplification 2, eq. (17)) and its transform
# ---------------------------------------------------------------------------------------

def test_jacobi_vs_lapack_and_2x2(O):
    S = np.random.default_rng(16).standard_normal((40, 40))
    S = S + S.T
    w, V = O.jacobi_eigh(S)
    wl, Vl = np.linalg.eigh(S)
    np.testing.assert_allclose(w, wl[::-1], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.abs(V.T @ Vl[:, ::-1]), np.eye(40), atol=1e-8)
    np.testing.assert_allclose(V @ np.diag(w) @ V.T, S, atol=1e-11)


def test_subspace_iteration_vs_lapack(O):
    from fac_whitening_gb300 import synth
    Q = synth.haar_orthogonal(400, 18, "cpu", torch.float64).numpy()
    ev = np.arange(1, 401, dtype=np.float64) ** -1.6
    A = (Q * ev) @ Q.T
    mu, U = O.subspace_iteration(lambda X: A @ X, 400, k=64, iters=16)
    np.testing.assert_allclose(mu[:32], ev[:32], rtol=1e-8)
    # residual bound ||A u - mu u|| small, orthonormal columns
    res = np.linalg.norm(A @ U[:, :32] - U[:, :32] * mu[:32], axis=0)
    assert np.all(res <= 1e-6 * mu[:32])
    np.testing.assert_allclose(U[:, :32].T @ U[:, :32], np.eye(32), atol=1e-12)


def test_lowrank_full_rank_whitens_exactly(O):
    # r = d_in: T_A^T A T_A = I, and T_A equals the symmetric A^-1/2 (LAPACK eigh)
    A = _spd(12, 19, 1e3)
    F = O.lowrank_factor_from_A(A, r=12)
    T = O.lowrank_T(F)
    np.testing.assert_allclose(T.T @ A @ T, np.eye(12), atol=1e-10)
    w, V = np.linalg.eigh(A)
    np.testing.assert_allclose(T, (V / np.sqrt(w)) @ V.T, atol=1e-9)


def test_lowrank_completion_properties(O):
    from fac_whitening_gb300 import synth
    rng = np.random.default_rng(20)
    a = synth.activations(600, 96, synth.spectrum_power_law(96, 1.0),
                          synth.haar_orthogonal(96, 21), 22).numpy()
    A = O.kfac_factor(a)
    F = O.lowrank_factor_from_A(A, r=32)
    Ah = F.dense()
    # sigma completion keeps the trace
    assert np.isclose(np.trace(Ah), np.trace(A), rtol=1e-12)
    # on span(U) the completed factor equals A (lambda = mu - sigma)
    np.testing.assert_allclose(Ah @ F.U, A @ F.U, atol=1e-10 * np.max(F.mu))
    # mu are the top eigenvalues of A (LAPACK)
    np.testing.assert_allclose(F.mu, np.sort(np.linalg.eigvalsh(A))[::-1][:32], rtol=1e-10)
    T, Ti = O.lowrank_T(F), O.lowrank_T(F, inverse=True)
    np.testing.assert_allclose(T @ Ti, np.eye(96), atol=1e-10)
    np.testing.assert_allclose(T.T @ Ah @ T, np.eye(96), atol=1e-9)
    np.testing.assert_allclose(T, T.T, atol=1e-12)
    W = rng.standard_normal((5, 96))
    np.testing.assert_allclose(O.lowrank_whiten(W, F), W @ T, atol=1e-10)
    np.testing.assert_allclose(O.lowrank_unwhiten(W, F), W @ Ti, atol=1e-10)
    # the activation route gives the same factor (never forms A when d_in > 128)
    F2 = O.lowrank_factor_from_activations(a, r=32)
    np.testing.assert_allclose(F2.mu, F.mu, rtol=1e-10)
    assert np.isclose(F2.sigma, F.sigma, rtol=1e-10)


def test_lowrank_activation_route_large(O):
    from fac_whitening_gb300 import synth
    a = synth.activations(1024, 300, synth.spectrum_power_law(300, 1.0),
                          synth.haar_orthogonal(300, 23), 24).numpy()
    F = O.lowrank_factor_from_activations(a, r=32)
    ev = np.sort(np.linalg.eigvalsh(O.kfac_factor(a)))[::-1]
    np.testing.assert_allclose(F.mu, ev[:32], rtol=1e-9)
    assert np.isclose(F.sigma, np.mean(ev[32:]), rtol=1e-9)


def test_error_feedback_update(O):
    # Algorithm 1, geometry-aware branch: U~ = U + R; R <- U~ - Dequantize(Q(U~)).
    # deq and U~ are within a factor two of each other (or deq = 0), so the new
    # residual is exact: deq + R_new == U~ bit for bit.
    rng = np.random.default_rng(25)
    W = rng.standard_normal((16, 48))
    R0 = (rng.standard_normal((16, 48)) * 0.01).astype(np.float32)
    q, Ut, R1 = O.encode_layer(W, O.Xform("identity"), "e4m3", residual=R0)
    np.testing.assert_array_equal(Ut, (W.astype(np.float32) + R0).astype(np.float32))
    deq = O.dequantize_any(q, "e4m3")
    np.testing.assert_array_equal((deq + R1).astype(np.float32), Ut)


def test_fidelity_closed_forms(O):
    g = np.array([3.0, -4.0, 0.0, 12.0])
    f = O.fidelity(g, g)
    assert f["rel_l2"] == 0 and np.isclose(f["cos"], 1) and f["max_err"] == 0 and f["mse"] == 0
    f = O.fidelity(2 * g, g)
    assert np.isclose(f["rel_l2"], 1) and np.isclose(f["cos"], 1)
    assert f["max_err"] == 12 and np.isclose(f["mse"], 169 / 4)
    assert np.isclose(O.fidelity(-g, g)["cos"], -1)


# ---------------------------------------------------------------------------------------
# the worked 2x2 example (golden values printed on the page)
# ---------------------------------------------------------------------------------------

def test_toy_2x2_golden(O):
    gold = json.load(open(os.path.join(GOLDEN, "toy_2x2.json")))

    def tol(entry):
        return entry["tol"] if "tol" in entry else 0.5 * 10 ** -entry["decimals"]

    A = np.array(gold["A"], dtype=np.float64)
    w, V = O.jacobi_eigh(A)
    np.testing.assert_allclose(w, gold["eigenvalues"]["value"], atol=tol(gold["eigenvalues"]))
    np.testing.assert_allclose(np.abs(V), np.abs(np.array(gold["eigenvectors"]["value"])), atol=1e-12)
    L = O.cholesky(A)
    np.testing.assert_allclose(L, gold["L_A"]["value"], atol=tol(gold["L_A"]))
    Li = O.lower_inverse(L)
    np.testing.assert_allclose(Li, gold["L_A_inv"]["value"], atol=tol(gold["L_A_inv"]))
    g = np.array([gold["g"]], dtype=np.float64)               # one gradient row
    gt = O.chol_input_whiten(g, L)[0]                           # g~^T = g^T L_A^-T
    np.testing.assert_allclose(gt, gold["g_tilde"]["value"], atol=tol(gold["g_tilde"]))
    qg = O.toy_quantize(g[0])
    np.testing.assert_allclose(qg, gold["toy_quantized_g"]["value"], atol=tol(gold["toy_quantized_g"]))
    assert abs(np.linalg.norm(qg - g[0]) - gold["toy_error_g"]["value"]) <= tol(gold["toy_error_g"])
    qgt = O.toy_quantize(gt)
    np.testing.assert_allclose(qgt, gold["toy_quantized_g_tilde"]["value"],
                               atol=tol(gold["toy_quantized_g_tilde"]))
    e = qgt - gt
    assert abs(np.linalg.norm(e) - gold["toy_error_g_tilde"]["value"]) <= tol(gold["toy_error_g_tilde"])
    back = O.chol_input_unwhiten(e[None, :], L)[0]             # eq. (14): error mapped back
    assert (np.linalg.norm(back) < gold["toy_error_g"]["value"]) == gold["mapped_back_error_smaller"]["value"]
