"""GPU parity of the rank-r whitening codec (simplification 2, eq. (17)) against the oracle.

The factor (U, mu, sigma) is the oracle's, rounded to FP32 and given to both sides.
Transforms and decoded tensors: relative Frobenius error <= 1e-5 (FP32 path).
Codes: bit-exact when the oracle quantises the GPU's transformed tensor; against
the oracle's own transformed tensor, codes may differ only where the two FP32
values straddle a rounding boundary (by one code step, on a tiny fraction)."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G
from fac_whitening_gb300 import synth

from gpu_util import DEV, ctx, encode, factor_to_gpu, rel_fro, status, t, ws

pytestmark = pytest.mark.gpu
TOL = 1e-5


def make_layer(d_out, d_in, T, exponent, seed, rank=32, R=1, dtype=torch.float32, device="cpu"):
    spec = synth.LayerSpec("t", d_out, d_in, T=T, exponent=exponent, act_dtype=dtype)
    Ws, a = synth.layer_inputs(spec, 9, seed, R, device=device)
    a64 = a.to(torch.float64).cpu().numpy()
    F = O.lowrank_factor_from_activations(a64, r=rank)
    F32 = O.LowRankFactor(F.U.astype(np.float32), F.mu.astype(np.float32), np.float32(F.sigma))
    return [W.cpu().numpy() for W in Ws], F32, a


def oracle_codes_close(out, want, fmt, scaling):
    """Codes from the GPU's transform against codes from the oracle's transform.

    Each side is round-to-nearest of its own input (checked bit-exactly elsewhere), and
    the inputs differ by the transform error, so where the codes differ the dequantised
    values may differ by at most that input difference plus one code spacing on each
    side; and they may differ only on a small fraction of the elements."""
    qg = O.quantize(out["tout"], fmt, scaling)
    qo = O.quantize(want.astype(np.float32), fmt, scaling)
    if fmt == "nvfp4":
        cg, co = qg["codes"], qo["codes"]
        diff = np.stack([cg & 0xF, cg >> 4], -1) != np.stack([co & 0xF, co >> 4], -1)
        assert np.count_nonzero(diff) / diff.size < 2e-3
        return
    diff = qg["codes"] != qo["codes"]
    assert np.count_nonzero(diff) / diff.size < 2e-3
    dg = O.dequantize_any(qg, fmt, scaling).astype(np.float64)
    do = O.dequantize_any(qo, fmt, scaling).astype(np.float64)
    f = O.FORMATS[fmt]
    if scaling == "tensor":
        s = np.full(dg.shape, float(max(qg["scales"][0], qo["scales"][0])))
    else:
        s = np.maximum(np.kron(qg["scales"], np.ones((128, 128))), np.kron(qo["scales"], np.ones((128, 128))))
        s = s[: dg.shape[0], : dg.shape[1]]
    spacing = np.maximum(np.abs(dg), np.abs(do)) * 2.0 ** -f.mbits + f.min_subnormal * s
    dx = np.abs(out["tout"].astype(np.float64) - want)
    assert np.all(np.abs(dg - do)[diff] <= (dx + 2 * spacing)[diff] * 1.0001)


@pytest.fixture(scope="module")
def tiny():
    return make_layer(64, 256, 512, 1.0, 0, R=4)


@pytest.fixture(scope="module")
def c3():
    # a 600M-like fc2 layer, 1536 x 6144, with the factor from 4096 tokens
    return make_layer(1536, 6144, 4096, 1.2, 1, R=1, dtype=torch.bfloat16, device="cuda")


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("e5m2", "tensor"), ("e4m3", "block128"),
                                         ("nvfp4", "tensor")])
@pytest.mark.parametrize("which", ["tiny", "c3"])
def test_lowrank_encode(which, fmt, scaling, request):
    Ws, F, _ = request.getfixturevalue(which)
    W = Ws[0]
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    out = encode(f, W, fmt, scaling)
    assert out["status"] == 0
    want = O.lowrank_whiten(W, F)
    assert rel_fro(out["tout"], want) <= TOL
    qg = O.quantize(out["tout"], fmt, scaling)                 # the quantiser contract, bit-exact
    np.testing.assert_array_equal(out["codes"], qg["codes"])
    np.testing.assert_array_equal(out["scales"], qg["scales"])
    oracle_codes_close(out, want, fmt, scaling)                # against the oracle's own transform


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("nvfp4", "tensor"), ("e5m2", "block128")])
def test_lowrank_encode_tc_precision(c3, fmt, scaling):
    # reduced-precision tensor-core path: transform within 2e-2, quantiser contract bit-exact
    Ws, F, _ = c3
    W = Ws[0]
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    out = encode(f, W, fmt, scaling, prec="tc")
    want = O.lowrank_whiten(W, F)
    err = rel_fro(out["tout"], want)
    assert err <= 2e-2, err
    qg = O.quantize(out["tout"], fmt, scaling)
    np.testing.assert_array_equal(out["codes"], qg["codes"])


def test_lowrank_error_feedback(tiny):
    Ws, F, _ = tiny
    W = Ws[1]
    R0 = (0.01 * np.random.default_rng(2).standard_normal(W.shape)).astype(np.float32)
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    out = encode(f, W, "e4m3", residual=R0)
    Ut = out["tout"]
    assert rel_fro(Ut, (O.lowrank_whiten(W, F) + R0)) <= TOL
    q = O.quantize(Ut, "e4m3")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["residual"], (Ut - O.dequantize_any(q, "e4m3")).astype(np.float32))


@pytest.mark.parametrize("which", ["tiny", "c3"])
def test_lowrank_decode_and_roundtrip(which, request):
    Ws, F, _ = request.getfixturevalue(which)
    W = Ws[0]
    d_out, d_in = W.shape
    f = factor_to_gpu("lowrank", d_out, d_in, F=F)
    X = np.random.default_rng(3).standard_normal(W.shape).astype(np.float32)
    Wo = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    st = status()
    w = ws("decode", "lowrank", "f32", "tensor", d_out, d_in)
    G.gift_decode(ctx(), f, t(X), False, "f32", "tensor", d_out, d_in, Wo, ws=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert rel_fro(Wo.cpu().numpy(), O.lowrank_unwhiten(X, F)) <= TOL
    # lossless format: map back inverts the whitening (common confusions: lossless GIFT == baseline).
    # Each direction is within 1e-5 of the oracle; the composition is not: whitening cancels
    # sigma^-1/2 W against the rank-r term, so one FP32 rounding (u = 2^-24) of that term
    # comes back multiplied by sqrt(mu_1 / sigma) in the map back.  Bound: 1e-5 + 8 u sqrt(mu_1/sigma).
    enc = encode(f, W, "f32")
    G.gift_decode(ctx(), f, enc["_dev"][0], False, "f32", "tensor", d_out, d_in, Wo, ws=w)
    torch.cuda.synchronize()
    tol_rt = TOL + 8 * 2.0 ** -24 * np.sqrt(float(F.mu[0]) / float(F.sigma))
    assert rel_fro(Wo.cpu().numpy(), W) <= tol_rt
    # decode straight from codes = dequantise then map back
    e8 = encode(f, W, "e4m3")
    G.gift_decode(ctx(), f, e8["_dev"][0], True, "e4m3", "tensor", d_out, d_in, Wo, scales=e8["_dev"][1], ws=w)
    torch.cuda.synchronize()
    deq = O.dequantize_any(O.quantize(e8["tout"], "e4m3"), "e4m3")
    assert rel_fro(Wo.cpu().numpy(), O.lowrank_unwhiten(deq, F)) <= TOL


def test_lowrank_reduce_decode_pipeline(tiny):
    Ws, F, _ = tiny
    d_out, d_in = Ws[0].shape
    f = factor_to_gpu("lowrank", d_out, d_in, F=F)
    outs = [encode(f, W, "e4m3") for W in Ws]
    avg = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    G.gift_replica_reduce(ctx(), [o["_dev"][0] for o in outs], [o["_dev"][1] for o in outs], "e4m3", "tensor",
                          d_out, d_in, avg)
    torch.cuda.synchronize()
    qs = [O.quantize(o["tout"], "e4m3") for o in outs]
    np.testing.assert_array_equal(avg.cpu().numpy(), O.replica_reduce(qs, "e4m3"))


@pytest.mark.parametrize("rank,d_in", [(8, 256), (16, 16), (1, 40)])
def test_lowrank_small_ranks(rank, d_in):
    rng = np.random.default_rng(4)
    a = rng.standard_normal((300, d_in)) * np.linspace(3, 0.2, d_in)
    F = O.lowrank_factor_from_A(O.kfac_factor(a), r=rank)
    F = O.LowRankFactor(F.U.astype(np.float32), F.mu.astype(np.float32), np.float32(F.sigma))
    W = rng.standard_normal((50, d_in)).astype(np.float32)
    f = factor_to_gpu("lowrank", 50, d_in, F=F)
    out = encode(f, W, "e4m3")
    assert rel_fro(out["tout"], O.lowrank_whiten(W, F)) <= TOL
    np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e4m3")["codes"])


@pytest.mark.parametrize("which,prec,fmt", [("tiny", "fp32", "e4m3"), ("c3", "fp32", "e4m3"), ("c3", "tc", "e4m3"),
                                             ("c3", "fp32", "nvfp4")])
def test_lowrank_amax_matches_transformed(which, prec, fmt, request):
    # gift_amax returns exactly the amax of the tensor gift_encode quantises (same kernel and
    # arithmetic for the shape), so a shared amax taken with it never clips an encode
    Ws, F, _ = request.getfixturevalue(which)
    W = Ws[-1]
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    acc = torch.zeros(1, dtype=torch.float32, device=DEV)
    G.gift_amax(ctx(), f, t(W), fmt, "tensor", acc, prec=prec, ws=ws("amax", "lowrank", fmt, "tensor", *W.shape))
    torch.cuda.synchronize()
    out = encode(f, W, fmt, prec=prec)
    assert acc.item() == np.max(np.abs(out["tout"])) == out["amax"][0]


@pytest.mark.parametrize("fmt", ["e4m3", "nvfp4"])
@pytest.mark.parametrize("prec", ["fp32", "tc"])
def test_cached_u_planes_match_per_call(c3, fmt, prec):
    # a factor carrying its U term planes (gift_factor_prepare) gives bit-identical encodes and
    # decodes to the same factor without them (planes rebuilt inside every call)
    Ws, F, _ = c3
    W = Ws[0]
    d_out, d_in = W.shape
    f0 = factor_to_gpu("lowrank", d_out, d_in, F=F)
    f1 = factor_to_gpu("lowrank", d_out, d_in, F=F)
    f1.planes = torch.zeros(G.lib().gift_factor_planes_bytes(d_in), dtype=torch.uint8, device=DEV)
    G.gift_factor_prepare(ctx(), f1)
    e0, e1 = encode(f0, W, fmt, prec=prec), encode(f1, W, fmt, prec=prec)
    assert e0["status"] == e1["status"] == 0
    np.testing.assert_array_equal(e0["codes"], e1["codes"])
    np.testing.assert_array_equal(e0["scales"], e1["scales"])
    np.testing.assert_array_equal(e0["tout"], e1["tout"])
    X = t(np.random.default_rng(4).standard_normal(W.shape).astype(np.float32))
    w = ws("decode", "lowrank", "f32", "tensor", d_out, d_in)
    outs = []
    for f in (f0, f1):
        Wo = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
        G.gift_decode(ctx(), f, X, False, "f32", "tensor", d_out, d_in, Wo, prec=prec, ws=w)
        torch.cuda.synchronize()
        outs.append(Wo.cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])


def test_factor_update_fills_planes():
    # gift_factor_update writes the planes together with U; they equal gift_factor_prepare's
    spec = synth.LayerSpec("m", 128, 1024, T=2048, exponent=1.0, act_dtype=torch.bfloat16)
    _, a = synth.layer_inputs(spec, 9, 4, 1, device="cuda")
    f = G.Factor.empty("lowrank", 128, 1024, 32, device=DEV, planes=True)
    n = G.gift_workspace_bytes(ctx(), "factor_update", "lowrank", "e4m3", "tensor", 128, 1024, a.shape[0])
    G.gift_factor_update(ctx(), f, a, seed=3, ws=torch.zeros(n, dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    got = f.planes.clone()
    f.planes.zero_()
    G.gift_factor_prepare(ctx(), f)
    torch.cuda.synchronize()
    assert torch.equal(got, f.planes) and int(got.count_nonzero()) > 0


@pytest.fixture(scope="module")
def ragged():
    # 200 rows: the last 128-row block is clipped; d_in 512 keeps the tensor-core apply
    return make_layer(200, 512, 1024, 1.0, 3, R=1)


@pytest.mark.parametrize("fmt,scaling", [("e4m3", "tensor"), ("nvfp4", "tensor"), ("e5m2", "block128"),
                                         ("e4m3", "block128")])
@pytest.mark.parametrize("which", ["c3", "ragged"])
def test_lowrank_error_feedback_formats(which, fmt, scaling, request):
    # error feedback through the tensor-core apply (Algorithm 1: U~ = W~ + R, then
    # R <- U~ - deq(Q(U~))): U~ within the transform tolerance of the oracle's, and the codes,
    # scales and new residual bit-exact against the oracle's quantiser applied to the GPU's U~
    Ws, F, _ = request.getfixturevalue(which)
    W = Ws[0]
    R0 = (0.3 * np.std(W) * np.random.default_rng(5).standard_normal(W.shape)).astype(np.float32)
    f = factor_to_gpu("lowrank", *W.shape, F=F)
    out = encode(f, W, fmt, scaling, residual=R0)
    assert out["status"] == 0
    Ut = out["tout"]
    assert rel_fro(Ut, O.lowrank_whiten(W, F) + R0) <= TOL
    q = O.quantize(Ut, fmt, scaling)
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["scales"], q["scales"])
    np.testing.assert_array_equal(out["residual"], (Ut.astype(np.float64) - O.dequantize_any(q, fmt, scaling))
                                  .astype(np.float32))


@pytest.mark.parametrize("which", ["c3", "ragged", "tiny"])
def test_lowrank_block_amax_matches_transformed(which, request):
    # gift_amax with 128 x 128 blocks returns each block's amax of exactly the tensor that
    # gift_encode quantises
    Ws, F, _ = request.getfixturevalue(which)
    W = Ws[-1]
    d_out, d_in = W.shape
    f = factor_to_gpu("lowrank", d_out, d_in, F=F)
    nb = ((d_out + 127) // 128) * ((d_in + 127) // 128)
    acc = torch.zeros(nb, dtype=torch.float32, device=DEV)
    G.gift_amax(ctx(), f, t(W), "e4m3", "block128", acc, ws=ws("amax", "lowrank", "e4m3", "block128", d_out, d_in))
    torch.cuda.synchronize()
    out = encode(f, W, "e4m3", "block128")
    got = acc.cpu().numpy()
    np.testing.assert_array_equal(got, out["amax"])
    np.testing.assert_array_equal(got.reshape(out["scales"].shape), O.block_amax(out["tout"]))


def test_lowrank_block_unaligned_simt():
    # d_in not a multiple of 128: the FP32-SIMT apply, same contract
    rng = np.random.default_rng(6)
    a = rng.standard_normal((600, 288)) * np.linspace(3, 0.2, 288)
    F = O.lowrank_factor_from_A(O.kfac_factor(a), r=32)
    F = O.LowRankFactor(F.U.astype(np.float32), F.mu.astype(np.float32), np.float32(F.sigma))
    W = rng.standard_normal((200, 288)).astype(np.float32)
    R0 = (0.1 * rng.standard_normal(W.shape)).astype(np.float32)
    f = factor_to_gpu("lowrank", 200, 288, F=F)
    out = encode(f, W, "e4m3", "block128", residual=R0)
    assert rel_fro(out["tout"], O.lowrank_whiten(W, F) + R0) <= TOL
    q = O.quantize(out["tout"], "e4m3", "block128")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    np.testing.assert_array_equal(out["residual"], (out["tout"].astype(np.float64) - O.dequantize_any(q, "e4m3", "block128"))
                                  .astype(np.float32))


@pytest.mark.parametrize("sms", [38, 7])
def test_reduced_sm_context(c3, sms):
    # a context sized for a share of the SMs (GIFT_OPT_SMS, for calls run side by side on
    # several streams) keeps the contract: encode within the transform tolerance with codes
    # that quantise its own W~, decode within 1e-5 of the oracle's map back
    Ws, F, _ = c3
    W = Ws[0]
    d_out, d_in = W.shape
    cq = G.Context(torch.cuda.current_device())
    G.gift_set_option(cq, G.OPT_SMS, sms)
    f = factor_to_gpu("lowrank", d_out, d_in, F=F)
    codes, scales, _ = (torch.empty(d_out * d_in, dtype=torch.uint8, device=DEV), torch.empty(1, device=DEV), None)
    tout = torch.empty(d_out, d_in, device=DEV)
    st = status()
    wenc = torch.zeros(G.gift_workspace_bytes(cq, "encode", "lowrank", "e4m3", "tensor", d_out, d_in),
                       dtype=torch.uint8, device=DEV)
    G.gift_encode(cq, f, t(W), "e4m3", "tensor", codes, scales, transformed_out=tout, ws=wenc, status=st)
    X = np.random.default_rng(9).standard_normal(W.shape).astype(np.float32)
    Wo = torch.empty(d_out, d_in, device=DEV)
    wdec = torch.zeros(G.gift_workspace_bytes(cq, "decode", "lowrank", "f32", "tensor", d_out, d_in),
                       dtype=torch.uint8, device=DEV)
    G.gift_decode(cq, f, t(X), False, "f32", "tensor", d_out, d_in, Wo, ws=wdec, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    tw = tout.cpu().numpy()
    assert rel_fro(tw, O.lowrank_whiten(W, F)) <= TOL
    np.testing.assert_array_equal(codes.cpu().numpy().reshape(W.shape), O.quantize(tw, "e4m3")["codes"])
    assert rel_fro(Wo.cpu().numpy(), O.lowrank_unwhiten(X, F)) <= TOL
    with pytest.raises(G.GiftError):
        G.gift_set_option(cq, G.OPT_SMS, 100000)
