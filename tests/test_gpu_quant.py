"""GPU parity of the Euclidean (identity-transform) codec path against the CPU oracle.

Codes, scales, residuals, reduced averages and hit counts are integer or exactly
rounded results: they must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G

from gpu_util import DEV, alloc_codes, ctx, encode, status, t, ws

pytestmark = pytest.mark.gpu
FMAX = {"e4m3": 448.0, "e5m2": 57344.0}


def probe(fmt):
    """Every midpoint between adjacent codes, one FP32 ulp either side, the codes themselves."""
    vals = np.unique(np.abs(O.decode(np.arange(128), O.FORMATS[fmt])))
    vals = vals[np.isfinite(vals)]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    pts = np.concatenate([vals.astype(np.float32), mids, np.nextafter(mids, np.float32(np.inf)),
                          np.nextafter(mids, np.float32(-np.inf)),
                          np.float32([FMAX[fmt] * 1.03, FMAX[fmt] * 40, 1e-30, 1e-45, 0])])
    return np.concatenate([pts, -pts]).astype(np.float32)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_rounding_midpoints_and_random_bits(fmt):
    # with amax = FMAX the multiplier is exactly 1, so the codes are the hardware rounding of x
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    rnd = bits.view(np.float32)
    rnd = rnd[np.isfinite(rnd)]
    x = np.concatenate([probe(fmt), rnd]).astype(np.float32)
    x = x[: (len(x) // 4) * 4].reshape(4, -1)
    out = encode(None, x, fmt, amax_in=np.float32(FMAX[fmt]))
    np.testing.assert_array_equal(out["codes"], O.quantize(x, fmt, amax=FMAX[fmt])["codes"])


@pytest.mark.parametrize("shape", [(64, 256), (37, 53), (1536, 6144)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_tensor(shape, fmt):
    rng = np.random.default_rng(2)
    W = (rng.standard_normal(shape) * np.exp(rng.uniform(-3, 3, shape[1]))).astype(np.float32)
    out = encode(None, W, fmt)
    q = O.quantize(W, fmt)
    assert out["status"] == 0
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
    assert out["amax"][0] == q["amax"]
    np.testing.assert_array_equal(out["tout"], W)


def test_encode_unaligned_scalar_path():
    rng = np.random.default_rng(3)
    base = torch.tensor(rng.standard_normal(64 * 33 + 1).astype(np.float32), device=DEV)
    Wt = base[1:].view(64, 33)                     # 4-byte aligned only
    out = encode(None, None, "e4m3", Wt=Wt)
    np.testing.assert_array_equal(out["codes"], O.quantize(Wt.cpu().numpy(), "e4m3")["codes"])


@pytest.mark.parametrize("shape", [(300, 200), (129, 131), (1536, 6144)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_block128(shape, fmt):
    rng = np.random.default_rng(4)
    W = (rng.standard_t(3, shape) * np.exp(2 * rng.standard_normal(shape[1]))).astype(np.float32)
    out = encode(None, W, fmt, "block128")
    q = O.quantize(W, fmt, "block128")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
    np.testing.assert_array_equal(out["amax"].reshape(q["amax"].shape), q["amax"])


@pytest.mark.parametrize("shape", [(48, 64), (5, 48), (1536, 6144)])
def test_encode_nvfp4(shape):
    rng = np.random.default_rng(5)
    W = (rng.standard_normal(shape) * np.exp(rng.uniform(-4, 4, (shape[0], 1)))).astype(np.float32)
    W[0, :16] = 0.0                                  # an all-zero group
    out = encode(None, W, "nvfp4")
    q = O.quantize(W, "nvfp4")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
    assert out["tensor_scale"] == q["tensor_scale"]


def test_encode_nvfp4_unaligned():
    rng = np.random.default_rng(6)
    base = torch.tensor(rng.standard_normal(16 * 32 + 1).astype(np.float32), device=DEV)
    Wt = base[1:].view(16, 32)
    out = encode(None, None, "nvfp4", Wt=Wt)
    q = O.quantize(Wt.cpu().numpy(), "nvfp4")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])


@pytest.mark.parametrize("fmt,scaling,shape", [("e4m3", "tensor", (64, 256)), ("e5m2", "block128", (200, 300)),
                                               ("nvfp4", "tensor", (32, 64)), ("e4m3", "tensor", (17, 19)),
                                               ("e4m3", "block512", (17, 19)), ("e5m2", "block512", (64, 256))])
def test_error_feedback(fmt, scaling, shape):
    rng = np.random.default_rng(7)
    W = rng.standard_normal(shape).astype(np.float32)
    R0 = (0.05 * rng.standard_normal(shape)).astype(np.float32)
    out = encode(None, W, fmt, scaling, residual=R0)
    q, Ut, R1 = O.encode_layer(W, O.Xform("identity"), fmt, scaling, residual=R0)
    np.testing.assert_array_equal(out["tout"], Ut)
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["residual"], R1)


def test_zero_tensor_and_nonfinite_status():
    Z = np.zeros((8, 64), np.float32)
    Z[0, 0] = -0.0
    out = encode(None, Z, "e4m3")
    np.testing.assert_array_equal(out["codes"], O.quantize(Z, "e4m3")["codes"])
    assert out["scales"][0] == 0 and out["status"] == 0
    bad = np.ones((8, 64), np.float32)
    bad[3, 5] = np.nan
    assert encode(None, bad, "e4m3")["status"] == G.ERR_NONFINITE
    bad[3, 5] = np.inf
    assert encode(None, bad, "e5m2", "block128")["status"] == G.ERR_NONFINITE


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("e5m2", "block128"), ("nvfp4", "tensor"),
                                         ("e4m3", "block512")])
def test_shared_amax_euclidean_path(fmt, scaling):
    # Algorithm 1, Euclidean path: Scale, AllReduceMax, Q with the shared scale
    rng = np.random.default_rng(8)
    Ws = [(rng.standard_normal((130, 256)) * (1 + r)).astype(np.float32) for r in range(4)]
    nblk = 1 if scaling == "tensor" or fmt == "nvfp4" else (2 * 2 if scaling == "block128" else 65)
    acc = torch.zeros(nblk, dtype=torch.float32, device=DEV)
    w = ws("amax", "identity", fmt, scaling, 130, 256)
    st = status()
    for W in Ws:
        G.gift_amax(ctx(), None, t(W), fmt, scaling, acc, ws=w, status=st)
    torch.cuda.synchronize()
    if scaling == "tensor" or fmt == "nvfp4":
        shared = np.float32(max(O.abs_max(W) for W in Ws))
        assert acc.item() == shared
    elif scaling == "block512":
        shared = np.maximum.reduce([O.quantize(W, fmt, "block512")["amax"] for W in Ws])
        np.testing.assert_array_equal(acc.cpu().numpy(), shared)
    else:
        shared = np.maximum.reduce([O.block_amax(W) for W in Ws])
        np.testing.assert_array_equal(acc.cpu().numpy().reshape(shared.shape), shared)
    for W in Ws:
        out = encode(None, W, fmt, scaling, amax_in=shared if np.ndim(shared) == 0 else shared.ravel())
        np.testing.assert_array_equal(out["codes"], O.quantize(W, fmt, scaling, amax=shared)["codes"])


@pytest.mark.parametrize("fmt,scaling,R,shape", [("e4m3", "tensor", 8, (64, 256)), ("e5m2", "block128", 3, (200, 300)),
                                                 ("e4m3", "block128", 4, (256, 384)), ("nvfp4", "tensor", 4, (48, 64)),
                                                 ("f32", "tensor", 4, (33, 35)), ("e4m3", "tensor", 5, (7, 9)),
                                                 ("e4m3", "block512", 4, (33, 47)),
                                                 ("e5m2", "block512", 3, (1536, 1536))])
def test_replica_reduce(fmt, scaling, R, shape):
    rng = np.random.default_rng(9)
    Ws = [(rng.standard_normal(shape) * (0.5 + r)).astype(np.float32) for r in range(R)]
    Ws[0][0, 0] = -0.0
    outs = [encode(None, W, fmt, scaling) for W in Ws]
    qs = [O.quantize(W, fmt, scaling) for W in Ws]
    avg = torch.empty(*shape, dtype=torch.float32, device=DEV)
    codes = [o["_dev"][0] for o in outs]
    scales = None if fmt == "f32" else [o["_dev"][1] for o in outs]
    tsc = [o["_dev"][2] for o in outs] if fmt == "nvfp4" else None
    G.gift_replica_reduce(ctx(), codes, scales, fmt, scaling, shape[0], shape[1], avg, tensor_scales=tsc)
    torch.cuda.synchronize()
    want = O.replica_reduce(qs, fmt, scaling)
    np.testing.assert_array_equal(avg.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("e5m2", "block128"), ("nvfp4", "tensor"),
                                         ("e4m3", "block512")])
def test_decode_identity_from_codes(fmt, scaling):
    rng = np.random.default_rng(10)
    W = rng.standard_normal((96, 160)).astype(np.float32)
    out = encode(None, W, fmt, scaling)
    codes, scales, tsc = out["_dev"]
    Wo = torch.empty(96, 160, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), None, codes, True, fmt, scaling, 96, 160, Wo, scales=scales, tensor_scale=tsc,
                  ws=ws("decode", "identity", fmt, scaling, 96, 160))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Wo.cpu().numpy(), O.dequantize_any(O.quantize(W, fmt, scaling), fmt, scaling))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scaling", ["tensor", "block128", "block512"])
@pytest.mark.parametrize("shape", [(1536, 1536), (300, 200), (6144, 1536)])
def test_boundary_hits(fmt, scaling, shape):
    from fac_whitening_gb300 import synth
    W = synth.student_t_colscaled(*shape, seed=11 + shape[0]).numpy()
    W[0, :7] = 0
    counts = torch.zeros(3, dtype=torch.int64, device=DEV)
    w = ws("amax", "identity", fmt, scaling, *shape)
    for _ in range(2):   # counts accumulate over a profiling window
        G.gift_boundary_hit_rate(ctx(), t(W), fmt, scaling, counts, ws=w)
    torch.cuda.synchronize()
    up, lo, n = O.boundary_hits(W, fmt, scaling)
    assert counts.cpu().tolist() == [2 * up, 2 * lo, 2 * n]


@pytest.mark.parametrize("shape", [(1536, 6144), (37, 101), (64, 256)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_block512(shape, fmt):
    # the per-block Euclidean baseline of the experiments: one scale per 512 consecutive
    # elements, the last block shorter (37 x 101 = 3737 elements: ragged, not a multiple of 4)
    from fac_whitening_gb300 import synth
    W = synth.student_t_colscaled(*shape, seed=31 + shape[0]).numpy()
    out = encode(None, W, fmt, "block512")
    q = O.quantize(W, fmt, "block512")
    assert out["status"] == 0
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
    np.testing.assert_array_equal(out["amax"], q["amax"])
    np.testing.assert_array_equal(out["tout"], W)


def test_encode_block512_unaligned_and_transforms():
    rng = np.random.default_rng(32)
    base = torch.tensor(rng.standard_normal(64 * 33 + 1).astype(np.float32), device=DEV)
    out = encode(None, None, "e5m2", "block512", Wt=base[1:].view(64, 33))   # 4-byte aligned only
    np.testing.assert_array_equal(out["codes"], O.quantize(base[1:].view(64, 33).cpu().numpy(), "e5m2",
                                                           "block512")["codes"])
    # a Cholesky transform followed by the block-512 pack
    from gpu_util import factor_to_gpu, rel_fro
    A = np.cov(rng.standard_normal((96, 400))) + 0.1 * np.eye(96)
    LA = O.cholesky(A).astype(np.float32)
    LAi = O.lower_inverse(LA).astype(np.float32)
    W = rng.standard_normal((40, 96)).astype(np.float32)
    f = factor_to_gpu("chol_input", 40, 96, LA=LA, LAinv=LAi)
    out = encode(f, W, "e4m3", "block512")
    assert rel_fro(out["tout"], O.Xform("chol_input", LA=LA, LAinv=LAi).whiten(W)) <= 1e-5
    np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e4m3", "block512")["codes"])
    # a rank-r factor has no block-512 path
    U = np.linalg.qr(rng.standard_normal((96, 8)))[0].astype(np.float32)
    F = O.LowRankFactor(U, np.linspace(4, 1, 8).astype(np.float32), np.float32(0.1))
    f = factor_to_gpu("lowrank", 40, 96, F=F)
    with pytest.raises(G.GiftError) as e:
        encode(f, W, "e4m3", "block512")
    assert e.value.status == G.ERR_UNSUPPORTED


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scaling", ["tensor", "block128"])
def test_boundary_hits_batched(fmt, scaling):
    # one call over tensors of different sizes (aligned, unaligned, a 1-element tensor, an
    # all-zero tensor, more than 64 tensors) gives exactly the per-tensor counts, and the oracle's
    rng = np.random.default_rng(31)
    shapes = [(300, 1024), (1, 1), (17, 33), (64, 256), (8, 8)] * 14   # 70 tensors
    Ws = [t(rng.standard_t(3, size=s).astype(np.float32) * np.exp(rng.normal(0, 2, size=(1, s[1]))).astype(np.float32))
          for s in shapes]
    Ws[4] = torch.zeros(8, 8, device=DEV)
    n = len(Ws)
    got = torch.zeros(n, 3, dtype=torch.int64, device=DEV)
    want = torch.zeros(n, 3, dtype=torch.int64, device=DEV)
    w = ws("amax", "identity", fmt, "tensor", 1, 1)
    st = status()
    G.gift_boundary_hit_rates(ctx(), Ws, fmt, scaling, got, ws=w, status=st)
    for i, W in enumerate(Ws):
        G.gift_boundary_hit_rate(ctx(), W, fmt, scaling, want[i], ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(got, want)
    for i in (0, 2, 4):
        up, lo, cnt = O.boundary_hits(Ws[i].cpu().numpy(), fmt, scaling)
        assert got[i].tolist() == [up, lo, cnt]
