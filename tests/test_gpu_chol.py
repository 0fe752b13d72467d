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
