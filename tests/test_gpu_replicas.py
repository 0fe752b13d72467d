"""gift_encode_replicas: the R data-parallel replicas of one layer encoded by one call.

Its contract is equality with R gift_encode calls on the same arguments (whose parity with
the oracle is checked in test_gpu_lowrank.py and test_gpu_codec.py), so every output is
compared bit for bit: codes, scales, NVFP4 tensor scales, the amax written back, status.
Shapes: the 600M-like fc2 layer (eight column tiles per CTA), the 300M-like fc2 layer (three
or four tiles per CTA), a ragged row count, and a narrow layer with one tile per CTA; more
than 16 replicas take two launches.

gift_encode_replicas_shared (one scale for all replicas) is checked against the oracle (the
max of the replicas' amax, each replica quantised with it) and, bit for bit, against the
three steps it stands for: a zeroed word, gift_amax_replicas into it, gift_encode_replicas
with it as every replica's amax."""
import numpy as np
import pytest
import torch

import oracle as O
from fac_whitening_gb300 import gift as G

from gpu_util import DEV, alloc_codes, ctx, status, t, ws

pytestmark = pytest.mark.gpu


def rand_factor(d_out, d_in, seed, rank=32, planes=False):
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((d_in, rank)))
    mu = np.sort(rng.uniform(0.5, 50.0, rank))[::-1].copy()
    f = G.Factor("lowrank", d_out, d_in, rank, U=t(U.astype(np.float32)), mu=t(mu.astype(np.float32)),
                 sigma=t([0.05]))
    if planes:
        f.planes = torch.zeros(G.lib().gift_factor_planes_bytes(d_in), dtype=torch.uint8, device=DEV)
        G.gift_factor_prepare(ctx(), f)
    return f


def replicas(f, R, seed):
    """R gradients with an isotropic part and a part in the factor's subspace (each replica
    its own draw), so that the whitening changes them."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    Ws = []
    for _ in range(R):
        W = torch.randn(f.d_out, f.d_in, generator=gen, device=DEV) * 0.1
        W += (torch.randn(f.d_out, f.rank, generator=gen, device=DEV) * 3.0) @ f.U.T
        Ws.append(W.contiguous())
    return Ws


def outputs(fmt, scaling, d_out, d_in, R):
    outs = []
    for _ in range(R):
        codes, scales, tscale = alloc_codes(fmt, scaling, d_out, d_in)
        codes.fill_(0xA5)
        outs.append({"codes": codes, "scales": scales, "tscale": tscale,
                     "amax": torch.full((1,), -1.0, device=DEV)})
    return outs


def run_single(f, Ws, fmt, scaling, prec, amax_in=None):
    d_out, d_in = Ws[0].shape
    kind = "identity" if f is None else f.kind
    w = ws("encode", kind, fmt, scaling, d_out, d_in)
    outs, st = outputs(fmt, scaling, d_out, d_in, len(Ws)), status()
    for r, W in enumerate(Ws):
        o = outs[r]
        G.gift_encode(ctx(), f, W, fmt, scaling, o["codes"], o["scales"], o["tscale"],
                      amax_in=None if amax_in is None else amax_in[r],
                      amax_out=o["amax"] if scaling == "tensor" else None, prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    return outs, int(st.item())


def run_batched(f, Ws, fmt, scaling, prec, amax_in=None):
    d_out, d_in = Ws[0].shape
    kind = "identity" if f is None else f.kind
    w = ws("encode", kind, fmt, scaling, d_out, d_in)
    outs, st = outputs(fmt, scaling, d_out, d_in, len(Ws)), status()
    G.gift_encode_replicas(ctx(), f, Ws, fmt, scaling, [o["codes"] for o in outs],
                           scales=[o["scales"] for o in outs],
                           tensor_scales=[o["tscale"] for o in outs] if fmt == "nvfp4" else None,
                           amax_in=amax_in, amax_out=[o["amax"] for o in outs] if scaling == "tensor" else None,
                           prec=prec, ws=w, status=st)
    torch.cuda.synchronize()
    return outs, int(st.item())


def assert_same(a, b):
    (oa, sa), (ob, sb) = a, b
    assert sa == sb == 0
    for x, y in zip(oa, ob):
        for key in ("codes", "scales", "tscale", "amax"):
            if x[key] is not None:
                assert torch.equal(x[key], y[key]), key
    # the replicas were really different tensors
    assert not torch.equal(oa[0]["codes"], oa[-1]["codes"])


SHAPES = [(1536, 6144), (1024, 4096), (1000, 4096), (384, 2112)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "nvfp4"])
@pytest.mark.parametrize("prec", ["fp32", "tc"])
def test_encode_replicas_match_single_calls(shape, fmt, prec):
    f = rand_factor(*shape, seed=11)
    Ws = replicas(f, 5, seed=21)
    assert_same(run_batched(f, Ws, fmt, "tensor", prec), run_single(f, Ws, fmt, "tensor", prec))


def test_encode_replicas_two_launches():
    # 17 replicas: a batch of 16 and a batch of 1, the workspace reused in stream order
    f = rand_factor(1536, 6144, seed=12)
    Ws = replicas(f, 17, seed=22)
    assert_same(run_batched(f, Ws, "e4m3", "tensor", "fp32"), run_single(f, Ws, "e4m3", "tensor", "fp32"))


@pytest.mark.parametrize("fmt", ["e4m3", "nvfp4"])
def test_encode_replicas_cached_planes_and_caller_amax(fmt):
    # a factor carrying its U term planes; a caller amax for some replicas (one grid barrier
    # fewer for those) and the tensor's own for the others
    f = rand_factor(1536, 6144, seed=13, planes=True)
    Ws = replicas(f, 6, seed=23)
    amax_in = [torch.full((1,), 40.0, device=DEV) if r % 2 else None for r in range(6)]
    a = run_batched(f, Ws, fmt, "tensor", "fp32", amax_in=[x if x is not None else 0 for x in amax_in])
    b = run_single(f, Ws, fmt, "tensor", "fp32", amax_in=amax_in)
    assert_same(a, b)
    assert a[0][1]["amax"].item() == 40.0 and a[0][0]["amax"].item() != 40.0


@pytest.mark.parametrize("case", ["identity", "block128", "f32"])
def test_encode_replicas_other_paths(case):
    # kinds and scalings outside the batched low-rank kernels: the same as per-replica calls
    f = None if case == "identity" else rand_factor(512, 2048, seed=14)
    fmt = "f32" if case == "f32" else "e4m3"
    scaling = "block128" if case == "block128" else "tensor"
    Ws = replicas(rand_factor(512, 2048, seed=14), 3, seed=24)
    assert_same(run_batched(f, Ws, fmt, scaling, "fp32"), run_single(f, Ws, fmt, scaling, "fp32"))


def test_encode_replicas_rejects_before_enqueueing():
    f = rand_factor(256, 1024, seed=15)
    Ws = replicas(f, 3, seed=25)
    w = ws("encode", "lowrank", "e4m3", "tensor", 256, 1024)
    outs = outputs("e4m3", "tensor", 256, 1024, 3)
    codes = [o["codes"] for o in outs]
    scales = [o["scales"] for o in outs]
    with pytest.raises(G.GiftError):   # replica 2 has no scale buffer
        G.gift_encode_replicas(ctx(), f, Ws, "e4m3", "tensor", codes, scales=scales[:2] + [0], ws=w)
    with pytest.raises(G.GiftError):   # replica 1 aliases its input
        G.gift_encode_replicas(ctx(), f, Ws, "e4m3", "tensor", [codes[0], Ws[1], codes[2]], scales=scales, ws=w)
    torch.cuda.synchronize()
    assert all(int((c != 0xA5).sum()) == 0 for c in codes)


@pytest.mark.parametrize("kind,shape", [("identity", (1536, 1536)), ("identity", (1000, 2048)),
                                        ("lowrank", (1536, 6144))])
def test_amax_replicas_matches_single_calls(kind, shape):
    # the shared amax of R replicas (one streaming pass) equals the max of R gift_amax calls
    fac = rand_factor(*shape, seed=16)
    f = None if kind == "identity" else fac
    Ws = replicas(fac, 5, seed=26)
    w = ws("amax", kind, "e4m3", "tensor", *shape)
    acc = torch.zeros(1, device=DEV)
    G.gift_amax_replicas(ctx(), f, Ws, "e4m3", "tensor", acc, ws=w)
    one = torch.zeros(1, device=DEV)
    for W in Ws:
        G.gift_amax(ctx(), f, W, "e4m3", "tensor", one, ws=w)
    torch.cuda.synchronize()
    assert acc.item() == one.item() > 0


def test_encode_replicas_identity_shared_amax():
    # the Euclidean path with a shared scale: one pack launch for all replicas
    fac = rand_factor(1536, 1536, seed=17)
    Ws = replicas(fac, 6, seed=27)
    shared = torch.zeros(1, device=DEV)
    G.gift_amax_replicas(ctx(), None, Ws, "e5m2", "tensor", shared, ws=ws("amax", "identity", "e5m2", "tensor", 1536, 1536))
    torch.cuda.synchronize()
    a = run_batched(None, Ws, "e5m2", "tensor", "fp32", amax_in=[shared] * 6)
    b = run_single(None, Ws, "e5m2", "tensor", "fp32", amax_in=[shared] * 6)
    assert_same(a, b)
    assert all(o["amax"].item() == shared.item() for o in a[0])


# ---- gift_encode_replicas_shared: one scale for all replicas (the synchronised amax) ----------

def shared_outputs(fmt, d_out, d_in, R):
    outs = outputs(fmt, "tensor", d_out, d_in, R)
    for o in outs:
        o["amax"] = None   # no per-replica amax copy in this call
    return outs


def run_shared(f, Ws, fmt, prec="fp32"):
    d_out, d_in = Ws[0].shape
    kind = "identity" if f is None else f.kind
    outs, st = shared_outputs(fmt, d_out, d_in, len(Ws)), status()
    shared = torch.full((1,), -1.0, device=DEV)
    G.gift_encode_replicas_shared(ctx(), f, Ws, fmt, "tensor", [o["codes"] for o in outs], [o["scales"] for o in outs],
                                  tensor_scales=[o["tscale"] for o in outs] if fmt == "nvfp4" else None,
                                  shared_amax_out=shared, prec=prec, ws=ws("encode", kind, fmt, "tensor", d_out, d_in),
                                  status=st)
    torch.cuda.synchronize()
    return outs, int(st.item()), shared.item()


def run_shared_steps(f, Ws, fmt, prec="fp32"):
    # the same result by its definition: a zeroed word, the replicas' amax max-accumulated
    # into it, then every replica encoded with that word as its amax
    d_out, d_in = Ws[0].shape
    kind = "identity" if f is None else f.kind
    word = torch.zeros(1, device=DEV)
    G.gift_amax_replicas(ctx(), f, Ws, fmt, "tensor", word, prec=prec, ws=ws("amax", kind, fmt, "tensor", d_out, d_in))
    outs, st = shared_outputs(fmt, d_out, d_in, len(Ws)), status()
    G.gift_encode_replicas(ctx(), f, Ws, fmt, "tensor", [o["codes"] for o in outs], scales=[o["scales"] for o in outs],
                           tensor_scales=[o["tscale"] for o in outs] if fmt == "nvfp4" else None,
                           amax_in=[word] * len(Ws), prec=prec, ws=ws("encode", kind, fmt, "tensor", d_out, d_in),
                           status=st)
    torch.cuda.synchronize()
    return outs, int(st.item()), word.item()


def spread_replicas(f, R, seed):
    # replicas whose own amax differ by orders of magnitude, so the shared scale is not theirs
    Ws = replicas(f, R, seed)
    for r, W in enumerate(Ws):
        W.mul_(10.0 ** (r % 4 - 1))
    return Ws


@pytest.mark.parametrize("shape", [(1536, 1536), (1536, 6144), (1000, 2048), (33, 35)], ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_shared_identity_matches_oracle(shape, fmt):
    # the fused launch (and, for 33x35, whose size is not a multiple of 4, the step sequence)
    # against the oracle: shared amax = max of the replicas' amax, each replica quantised with it
    fac = rand_factor(*shape, seed=31, rank=min(32, shape[1]))
    Ws = spread_replicas(fac, 8, seed=41)
    outs, st, shared = run_shared(None, Ws, fmt)
    assert st == 0
    host = [W.cpu().numpy() for W in Ws]
    amax = max(O.abs_max(x) for x in host)
    assert shared == amax
    for x, o in zip(host, outs):
        q = O.quantize(x, fmt, amax=amax)
        np.testing.assert_array_equal(o["codes"].cpu().numpy().reshape(x.shape), q["codes"])
        assert o["scales"].item() == q["scales"][0]
    # the small replicas really were coded with the large shared scale
    assert not np.array_equal(outs[0]["codes"].cpu().numpy().reshape(host[0].shape), O.quantize(host[0], fmt)["codes"])


@pytest.mark.parametrize("kind,fmt,prec", [("identity", "e4m3", "fp32"), ("identity", "nvfp4", "fp32"),
                                           ("lowrank", "e4m3", "fp32"), ("lowrank", "e5m2", "tc"),
                                           ("lowrank", "nvfp4", "fp32")])
def test_encode_shared_matches_steps(kind, fmt, prec):
    fac = rand_factor(1536, 6144, seed=32)
    f = None if kind == "identity" else fac
    Ws = spread_replicas(fac, 6, seed=42)
    (oa, sa, wa), (ob, sb, wb) = run_shared(f, Ws, fmt, prec), run_shared_steps(f, Ws, fmt, prec)
    assert sa == sb == 0 and wa == wb > 0
    for x, y in zip(oa, ob):
        for key in ("codes", "scales", "tscale"):
            if x[key] is not None:
                assert torch.equal(x[key], y[key]), key


def test_encode_shared_many_replicas_and_zeros():
    # 64 replicas (the maximum), some of them all zero; and all-zero replicas alone: amax 0,
    # scale 0, every code +0
    fac = rand_factor(256, 1024, seed=33)
    Ws = replicas(fac, 64, seed=43)
    for r in range(0, 64, 5):
        Ws[r].zero_()
    a, b = run_shared(None, Ws, "e4m3"), run_shared_steps(None, Ws, "e4m3")
    assert a[1] == b[1] == 0 and a[2] == b[2] > 0
    assert all(torch.equal(x["codes"], y["codes"]) and torch.equal(x["scales"], y["scales"])
               for x, y in zip(a[0], b[0]))
    Z = [torch.zeros(256, 1024, device=DEV) for _ in range(3)]
    outs, st, shared = run_shared(None, Z, "e5m2")
    assert st == 0 and shared == 0.0
    assert all(int(o["codes"].count_nonzero()) == 0 and o["scales"].item() == 0.0 for o in outs)


def test_encode_shared_nonfinite_and_rejects():
    fac = rand_factor(512, 2048, seed=34)
    Ws = replicas(fac, 4, seed=44)
    Ws[2][7, 9] = float("nan")
    assert run_shared(None, Ws, "e4m3")[1] == G.ERR_NONFINITE
    w = ws("encode", "identity", "e4m3", "block128", 512, 2048)
    outs = shared_outputs("e4m3", 512, 2048, 4)
    for fmt, scaling in (("e4m3", "block128"), ("f32", "tensor")):
        with pytest.raises(G.GiftError):
            G.gift_encode_replicas_shared(ctx(), None, Ws, fmt, scaling, [o["codes"] for o in outs],
                                          [o["scales"] for o in outs], ws=w)
