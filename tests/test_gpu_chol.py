"""GPU full-rank transforms (eqs. (11), (14), (16)) against the oracle, with the oracle's
Cholesky factors (and their inverses) rounded to FP32 and given to both sides."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G
from fac_whitening_gb300 import synth

from gpu_util import DEV, ctx, encode, factor_to_gpu, rel_fro, t, ws

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def layer():
    spec = synth.LayerSpec("c", 200, 384, T=3072, exponent=0.8, act_dtype=torch.float32)
    Ws, a = synth.layer_inputs(spec, 9, 5, 1)
    delta = synth.delta_for_layer(spec, 9, 5)
    LA = O.cholesky(O.kfac_factor(a.double().numpy()))
    LG = O.cholesky(O.kfac_factor(delta.double().numpy()))
    f32 = lambda x: x.astype(np.float32)   # noqa: E731
    return Ws[0].numpy(), f32(LA), f32(O.lower_inverse(LA)), f32(LG), f32(O.lower_inverse(LG))


@pytest.mark.parametrize("kind", ["chol_input", "chol_two_sided"])
def test_chol_encode_decode(layer, kind):
    W, LA, LAi, LG, LGi = layer
    d_out, d_in = W.shape
    f = factor_to_gpu(kind, d_out, d_in, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    xf = O.Xform(kind, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    out = encode(f, W, "e4m3")
    assert out["status"] == 0
    assert rel_fro(out["tout"], xf.whiten(W)) <= TOL
    np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e4m3")["codes"])
    X = np.random.default_rng(6).standard_normal(W.shape).astype(np.float32)
    Wo = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), f, t(X), False, "f32", "tensor", d_out, d_in, Wo,
                  ws=ws("decode", kind, "f32", "tensor", d_out, d_in))
    torch.cuda.synchronize()
    assert rel_fro(Wo.cpu().numpy(), xf.unwhiten(X)) <= TOL


@pytest.mark.parametrize("kind", ["chol_input", "chol_two_sided"])
def test_chol_tc_precision(layer, kind):
    # two BF16 terms and three products on the tensor cores: within 2e-2
    W, LA, LAi, LG, LGi = layer
    d_out, d_in = W.shape
    f = factor_to_gpu(kind, d_out, d_in, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    xf = O.Xform(kind, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    out = encode(f, W, "e4m3", prec="tc")
    assert out["status"] == 0
    assert rel_fro(out["tout"], xf.whiten(W)) <= 2e-2
    np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e4m3")["codes"])
    X = np.random.default_rng(7).standard_normal(W.shape).astype(np.float32)
    Wo = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), f, t(X), False, "f32", "tensor", d_out, d_in, Wo, prec="tc",
                  ws=ws("decode", kind, "f32", "tensor", d_out, d_in))
    torch.cuda.synchronize()
    assert rel_fro(Wo.cpu().numpy(), xf.unwhiten(X)) <= 2e-2


@pytest.mark.parametrize("variant", ["diagonal_A", "output_only"])
def test_ablation_variants_through_chol_kinds(layer, variant):
    # the ablations of simplifications 1 and 2 (Tables I and II): a diagonal input factor,
    # L_A = diag(sqrt(A_jj)), is CHOL_INPUT with a diagonal L_A; the output side only is
    # CHOL_TWO_SIDED with L_A = I
    W, LA, LAi, LG, LGi = layer
    d_out, d_in = W.shape
    if variant == "diagonal_A":
        dA = np.sqrt(np.sum(LA.astype(np.float64) ** 2, axis=1))   # sqrt of diag(L L^T) = sqrt(A_jj)
        LA, LAi = np.diag(dA).astype(np.float32), np.diag(1.0 / dA).astype(np.float32)
        kind = "chol_input"
    else:
        LA = LAi = np.eye(d_in, dtype=np.float32)
        kind = "chol_two_sided"
    f = factor_to_gpu(kind, d_out, d_in, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    xf = O.Xform(kind, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
    out = encode(f, W, "e4m3")
    assert out["status"] == 0
    assert rel_fro(out["tout"], xf.whiten(W)) <= TOL
    q = O.quantize(out["tout"], "e4m3")
    np.testing.assert_array_equal(out["codes"], q["codes"])
    X = O.dequantize_any(q, "e4m3")
    Wo = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    G.gift_decode(ctx(), f, t(X), False, "f32", "tensor", d_out, d_in, Wo,
                  ws=ws("decode", kind, "f32", "tensor", d_out, d_in))
    torch.cuda.synchronize()
    assert rel_fro(Wo.cpu().numpy(), xf.unwhiten(X)) <= TOL


def test_chol_ragged_shape():
    # d_out and d_in not multiples of the 128-row tiles nor of the 64-wide K chunks
    spec = synth.LayerSpec("r", 72, 150, T=600, exponent=1.0, act_dtype=torch.float32)
    Ws, a = synth.layer_inputs(spec, 9, 6, 1)
    delta = synth.delta_for_layer(spec, 9, 6)
    LA = O.cholesky(O.kfac_factor(a.double().numpy()))
    LG = O.cholesky(O.kfac_factor(delta.double().numpy()))
    f32 = lambda x: x.astype(np.float32)   # noqa: E731
    LA, LAi, LG, LGi = f32(LA), f32(O.lower_inverse(LA)), f32(LG), f32(O.lower_inverse(LG))
    W = Ws[0].numpy()
    for kind in ("chol_input", "chol_two_sided"):
        f = factor_to_gpu(kind, *W.shape, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
        xf = O.Xform(kind, LA=LA, LAinv=LAi, LG=LG, LGinv=LGi)
        out = encode(f, W, "e5m2")
        assert out["status"] == 0
        assert rel_fro(out["tout"], xf.whiten(W)) <= TOL
        np.testing.assert_array_equal(out["codes"], O.quantize(out["tout"], "e5m2")["codes"])
