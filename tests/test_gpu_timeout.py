"""The bounded waits end: a wait that runs out reports GIFT_ERR_TIMEOUT and the context
stays usable (no GPU fault, no hang).

The shared-scale encode (the AllReduceMax of Algorithm 1 followed by the pack, one
cooperative launch) waits at one grid-wide barrier with no asynchronous copy in flight.  With
the wait budget set to zero (GIFT_OPT_BARRIER_WAIT) a CTA that arrives before the others
gives up at once: it writes GIFT_ERR_TIMEOUT into the status word and stores no codes, and
the kernel ends.  The same context with the default budget then encodes correctly.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G

pytestmark = pytest.mark.gpu


def _shared_encode(ctx, Ws, st):
    d_out, d_in = Ws[0].shape
    codes = [torch.zeros(d_out * d_in, dtype=torch.uint8, device="cuda") for _ in Ws]
    scales = [torch.zeros(1, device="cuda") for _ in Ws]
    ws = torch.zeros(max(G.gift_workspace_bytes(ctx, "encode", "identity", "e4m3", "tensor", d_out, d_in), 256),
                     dtype=torch.uint8, device="cuda")
    G.gift_encode_replicas_shared(ctx, None, Ws, "e4m3", "tensor", codes, scales, ws=ws, status=st)
    torch.cuda.synchronize()
    return codes, scales


def test_barrier_wait_runs_out_and_context_survives():
    ctx = G.Context(torch.cuda.current_device())
    g = torch.Generator(device="cuda").manual_seed(5)
    Ws = [torch.randn(1536, 1536, generator=g, device="cuda") for _ in range(4)]
    with pytest.raises(G.GiftError):
        G.gift_set_option(ctx, G.OPT_BARRIER_WAIT, -1)
    G.gift_set_option(ctx, G.OPT_BARRIER_WAIT, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _shared_encode(ctx, Ws, st)
    assert int(st.item()) == G.ERR_TIMEOUT
    # the same context, default budget: the encode completes and matches the oracle
    G.gift_set_option(ctx, G.OPT_BARRIER_WAIT, 2_000_000_000)
    st.zero_()
    codes, scales = _shared_encode(ctx, Ws, st)
    assert int(st.item()) == 0
    Wn = [W.cpu().numpy() for W in Ws]
    amax = max(O.abs_max(W) for W in Wn)
    for W, c, s in zip(Wn, codes, scales):
        q = O.quantize(W, "e4m3", amax=amax)
        np.testing.assert_array_equal(c.cpu().numpy().reshape(W.shape), q["codes"])
        assert s.item() == q["scales"][0]
