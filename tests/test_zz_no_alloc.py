"""The allocation-free rank-r encode gives the same results as gift_encode.

gift_encode_lowrank_noalloc is for callers that cannot allocate device memory (for
example code running inside a gradient or communication hook while the framework's
allocator must not grow, or C callers without an allocator of their own): it keeps its
scratch in a fixed array inside the library instead of a caller workspace.  This test
calls it through the C ABI twice in a row (the second call must not see the first
call's scratch) and compares codes, scale and amax with gift_encode's (FP32 precision), bit
for bit, on every route the entry point takes: the batched tensor-core encode (the 600M-like
fc2 shape), the two-launch tensor-core apply (a shape whose row blocks do not fit the batched
plan), the FP32-SIMT path (d_in not a multiple of 32), and a caller-supplied amax.
The file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from fac_whitening_gb300 import gift as G

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    fn = G.lib().gift_encode_lowrank_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(G.GiftFactor), ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _factor(d_out, d_in, rank, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    q, _ = torch.linalg.qr(torch.randn(d_in, rank, generator=g, dtype=torch.float64))
    mu = torch.sort(torch.rand(rank, generator=g, dtype=torch.float64) * 10 + 1, descending=True).values
    # torch's QR returns a column-major Q; the library takes row-major, contiguous buffers
    f = G.Factor("lowrank", d_out, d_in, rank, U=q.float().contiguous().cuda(), mu=mu.float().cuda(),
                 sigma=torch.tensor([0.05], device="cuda"))
    return f


@pytest.mark.parametrize("shape,fmt,shared", [
    ((1536, 6144), "e4m3", False), ((1536, 6144), "e5m2", False), ((1536, 6144), "e4m3", True),
    ((4096, 4096), "e4m3", False), ((256, 1000), "e5m2", False), ((256, 1000), "e4m3", True)],
    ids=["600m-e4m3", "600m-e5m2", "600m-amax_in", "4096sq-e4m3", "simt-e5m2", "simt-amax_in"])
def test_noalloc_matches_gift_encode_twice(shape, fmt, shared):
    ctx = G.Context(torch.cuda.current_device())
    fn = _noalloc_fn()
    d_out, d_in = shape
    f = _factor(d_out, d_in, 32, 3)
    fs = f.c_struct()
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.zeros(G.gift_workspace_bytes(ctx, "encode", "lowrank", fmt, "tensor", d_out, d_in),
                     dtype=torch.uint8, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    for call in range(2):
        # the second tensor is much smaller, so a stale amax from the first call would show
        W = torch.randn(d_out, d_in, generator=g, device="cuda") * (1.0 if call == 0 else 1e-3)
        c_ref = torch.empty(d_out * d_in, dtype=torch.uint8, device="cuda")
        s_ref = torch.empty(1, dtype=torch.float32, device="cuda")
        a_ref = torch.empty(1, dtype=torch.float32, device="cuda")
        # a caller amax (the shared scale of the Euclidean path), below the tensor's own on the
        # first call (codes saturate) and above it on the second
        a_in = torch.tensor([3.0 if call == 0 else 0.25], device="cuda") if shared else None
        G.gift_encode(ctx, f, W, fmt, "tensor", c_ref, s_ref, amax_in=a_in, amax_out=a_ref, ws=ws)
        c = torch.empty_like(c_ref)
        s = torch.empty_like(s_ref)
        a = torch.empty_like(a_ref)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = fn(ctx.handle, ctypes.byref(fs), W.data_ptr(), d_out, d_in, G.FMT[fmt],
                None if a_in is None else a_in.data_ptr(), c.data_ptr(),
                s.data_ptr(), a.data_ptr(), st.data_ptr(), stream)
        assert rc == G.OK
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(a, a_ref) and torch.equal(s, s_ref)
        assert torch.equal(c, c_ref), int((c != c_ref).sum())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ctx = G.Context(torch.cuda.current_device())
    fn = _noalloc_fn()
    f = _factor(4097, 64, 8, 4)
    W = torch.zeros(4097, 64, device="cuda")
    c = torch.empty(4097 * 64, dtype=torch.uint8, device="cuda")
    s = torch.empty(1, device="cuda")
    rc = fn(ctx.handle, ctypes.byref(f.c_struct()), W.data_ptr(), 4097, 64, G.FMT["e4m3"], None, c.data_ptr(),
            s.data_ptr(), None, None, torch.cuda.current_stream().cuda_stream)
    assert rc == G.ERR_INVALID_ARG
