"""Seeded synthetic inputs for the GIFT gradient-codec workloads.

This module only *generates* inputs: random matrices, rotations, activations with
a chosen spectrum and the weight gradient of a linear layer formed from them.  It
holds none of the codec's arithmetic (no factor, transform, scale, quantiser,
reduction or decode), so that the CPU oracle and the CUDA path can both draw
their inputs from it without sharing any of the method.

The workloads stand in for the Llama-300M/600M pretraining gradients that the
GIFT pages measure on (GIFT reading notes, zhongzhuzhou.org, section
"Experimental setup"): the pages give no data, so every tensor here is drawn
from a seeded generator with the shape and statistics of the stated workload.

All generation runs in torch on the requested device.  The same seed gives the
same tensor on the same device type and torch build; tests never depend on the
CPU and CUDA streams agreeing, because both sides of a parity check always
receive the *same bytes* (generated once, then copied).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 0x61F7


def seed_for(config: int, layer: int = 0, replica: int = 0, stream: int = 0) -> int:
    """Seed of one tensor: workload id, layer, replica and a stream tag."""
    return SEED_BASE + 1000 * config + 17 * layer + replica + 7919 * stream


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def gaussian(shape, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """iid N(0, 1) entries."""
    g = _gen(seed, device)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)


_BASE_ROTATIONS = {}


def _base_rotation(n: int) -> torch.Tensor:
    """One Haar-distributed n x n orthogonal matrix per size (host QR, cached per process).

    QR of a Gaussian matrix with the signs of R's diagonal folded into Q (F. Mezzadri,
    "How to generate random matrices from the classical compact groups", Notices of
    the AMS, 2007).  Computed on the host so that no device linear-algebra library is
    needed; FP64 up to n = 2048, FP32 above.
    """
    if n not in _BASE_ROTATIONS:
        g = _gen(SEED_BASE + n, "cpu")
        work = torch.float64 if n <= 2048 else torch.float32
        z = torch.randn(n, n, generator=g, dtype=work)
        q, r = torch.linalg.qr(z)
        d = torch.sign(torch.diagonal(r))
        d[d == 0] = 1
        _BASE_ROTATIONS[n] = (q * d.unsqueeze(0)).contiguous()
    return _BASE_ROTATIONS[n]


def haar_orthogonal(n: int, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """A random orthogonal n x n matrix for `seed`: Q_base P D.

    Q_base is the per-size Haar matrix of _base_rotation; P is a seeded random column
    permutation and D seeded random signs, so every seed gives a different dense
    rotation (Q_base P D is orthogonal and, Q_base being Haar, Haar-distributed).
    """
    g = _gen(seed, "cpu")
    perm = torch.randperm(n, generator=g)
    signs = torch.randint(0, 2, (n,), generator=g).to(torch.float64) * 2 - 1
    q = _base_rotation(n)[:, perm] * signs.to(_base_rotation(n).dtype).unsqueeze(0)
    return q.to(device=device, dtype=dtype)


def spectrum_power_law(d: int, exponent: float, device="cpu") -> torch.Tensor:
    """s_i = i^-exponent, i = 1..d (column scales of the latent activations)."""
    i = torch.arange(1, d + 1, device=device, dtype=torch.float64)
    return i.pow(-float(exponent))


def spike_indices(d: int, count: int, seed: int) -> torch.Tensor:
    """`count` distinct seeded indices in [0, d) (CPU tensor)."""
    g = _gen(seed, "cpu")
    return torch.randperm(d, generator=g)[:count]


def activations(T: int, d_in: int, spectrum: torch.Tensor, Q: torch.Tensor, seed: int,
                device="cpu", dtype=torch.float32) -> torch.Tensor:
    """a = z diag(s) Q with z iid N(0,1) (T x d_in), rounded to `dtype`.

    The rows of `a` then have second moment Q^T diag(s^2) Q: an anisotropic
    input-activation cloud rotated away from the coordinate axes.
    """
    z = gaussian((T, d_in), seed, device, torch.float32)
    s = spectrum.to(device=device, dtype=torch.float32)
    a = (z * s.unsqueeze(0)) @ Q.to(device=device, dtype=torch.float32)
    return a.to(dtype)


def linear_layer_gradient(delta: torch.Tensor, a: torch.Tensor) -> torch.Tensor:
    """Weight gradient of a linear layer y = W a: W_g = delta^T a / T, in FP32.

    `delta` (T x d_out) and `a` (T x d_in) are widened exactly to FP32 first.
    """
    T = a.shape[0]
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        w = delta.to(torch.float32).t() @ a.to(torch.float32)
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return (w / T).contiguous()


def student_t_colscaled(d_out: int, d_in: int, seed: int, nu: int = 3, col_sigma: float = 2.0,
                        device="cpu") -> torch.Tensor:
    """Heavy-tailed gradient: Student-t(nu) entries times a per-column log-normal scale.

    t = z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared normals; the
    column scale is exp(N(0, col_sigma^2)).
    """
    g = _gen(seed, device)
    z = torch.randn(d_out, d_in, generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros(d_out, d_in, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi += torch.randn(d_out, d_in, generator=g, device=device, dtype=torch.float32).square()
    t = z / torch.sqrt(chi / nu)
    col = torch.exp(col_sigma * torch.randn(d_in, generator=g, device=device, dtype=torch.float32))
    return (t * col.unsqueeze(0)).contiguous()


# --------------------------------------------------------------------------------------
# Workload descriptions (shapes and statistics of the five synthetic workloads)
# --------------------------------------------------------------------------------------

@dataclass
class LayerSpec:
    name: str
    d_out: int
    d_in: int
    T: int = 0                 # tokens of activations (0: no activations, Euclidean tensor)
    exponent: float = 0.0      # spectrum exponent of the activations
    act_dtype: torch.dtype = torch.bfloat16
    spikes: int = 0            # number of x10 amplitude spikes in the spectrum
    kind: str = "gift"         # "gift" (geometry-aware branch) or "euclid"


@dataclass
class Workload:
    name: str
    config: int
    R: int
    layers: list = field(default_factory=list)


def tiny_workload() -> Workload:
    """Tiny single layer: W_g 64x256 from a 512x256 FP32 activation batch, R = 4."""
    return Workload("tiny-64x256", 0, 4,
                    [LayerSpec("tiny", 64, 256, T=512, exponent=1.0, act_dtype=torch.float32)])


def llama300m_fc2_workload() -> Workload:
    """Llama-300M-like MLP fc2: d_out 1024, d_in 4096, T 8192 BF16, spectrum i^-0.8, R = 8."""
    return Workload("llama300m-fc2-1024x4096", 1, 8,
                    [LayerSpec("fc2", 1024, 4096, T=8192, exponent=0.8)])


def llama600m_selective_workload(seed_layers: int = 13, euclid_each: int = 30) -> Workload:
    """Llama-600M-like selective deployment.

    13 fc2 layers 1536x6144 (T = 16384 BF16 activations, spectrum exponent drawn
    U[0.5, 1.2] per layer) take the geometry-aware branch; 60 Gaussian tensors,
    alternating 1536x1536 and 1536x6144, take the Euclidean path.  R = 8.
    """
    g = _gen(seed_for(2, stream=99), "cpu")
    exps = (0.5 + 0.7 * torch.rand(seed_layers, generator=g, dtype=torch.float64)).tolist()
    layers = [LayerSpec(f"fc2.{i}", 1536, 6144, T=16384, exponent=exps[i]) for i in range(seed_layers)]
    for j in range(2 * euclid_each):
        d_in = 1536 if j % 2 == 0 else 6144
        layers.append(LayerSpec(f"euclid.{j}", 1536, d_in, kind="euclid"))
    return Workload("llama600m-selective-13x1536x6144+60", 2, 8, layers)


def profiler_workload() -> Workload:
    """48 heavy-tailed gradients, 16 each of 1536x1536, 1536x6144 and 6144x1536."""
    shapes = [(1536, 1536), (1536, 6144), (6144, 1536)]
    layers = [LayerSpec(f"g{i}", *shapes[i % 3], kind="profile") for i in range(48)]
    return Workload("profiler-48-student-t", 3, 1, layers)


def stress_workload() -> Workload:
    """24 fc2-like layers 4096x16384, T = 32768 BF16, spectrum i^-1 with 8 x10 spikes, R = 16."""
    layers = [LayerSpec(f"fc2.{i}", 4096, 16384, T=32768, exponent=1.0, spikes=8) for i in range(24)]
    return Workload("stress-24x4096x16384", 4, 16, layers)


def layer_spectrum(spec: LayerSpec, config: int, layer: int, device="cpu") -> torch.Tensor:
    s = spectrum_power_law(spec.d_in, spec.exponent, device="cpu")
    if spec.spikes:
        idx = spike_indices(spec.d_in, spec.spikes, seed_for(config, layer, stream=5))
        s[idx] *= 10.0
    return s.to(device)


def layer_inputs(spec: LayerSpec, config: int, layer: int, R: int, device="cpu",
                 want_activations: bool = True):
    """Per-layer inputs: the replica gradients W_r and replica 0's activations a.

    Geometry-aware layers: Q (shared by the replicas of one layer) rotates the
    power-law spectrum; each replica r draws its own z and delta and its
    gradient is W_r = delta_r^T a_r / T.  Euclidean tensors: iid N(0,1) entries.
    Returns (list of R FP32 gradients, activations of replica 0 or None).
    """
    if spec.kind == "euclid":
        Ws = [gaussian((spec.d_out, spec.d_in), seed_for(config, layer, r), device) for r in range(R)]
        return Ws, None
    if spec.kind == "profile":
        return [student_t_colscaled(spec.d_out, spec.d_in, seed_for(config, layer, r), device=device)
                for r in range(R)], None
    Q = haar_orthogonal(spec.d_in, seed_for(config, layer, stream=1), device=device)
    s = layer_spectrum(spec, config, layer, device)
    Ws, a0 = [], None
    for r in range(R):
        a = activations(spec.T, spec.d_in, s, Q, seed_for(config, layer, r, stream=2), device,
                        spec.act_dtype)
        delta = gaussian((spec.T, spec.d_out), seed_for(config, layer, r, stream=3), device,
                         spec.act_dtype)
        Ws.append(linear_layer_gradient(delta, a))
        if r == 0:
            a0 = a if want_activations else None
        del delta
        if r != 0:
            del a
    return Ws, a0


def delta_for_layer(spec: LayerSpec, config: int, layer: int, replica: int = 0,
                    device="cpu") -> torch.Tensor:
    """The output-gradient batch delta (T x d_out) of one replica (two-sided factor G)."""
    return gaussian((spec.T, spec.d_out), seed_for(config, layer, replica, stream=3), device,
                    spec.act_dtype)


def random_omega_free_matrix(n: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    """iid N(0,1) n x k matrix (generic test matrix)."""
    return gaussian((n, k), seed, device)


def spd_matrix(n: int, cond: float, seed: int, dtype=torch.float64) -> torch.Tensor:
    """A symmetric positive definite n x n matrix with eigenvalues log-spaced in [1/cond, 1]."""
    Q = haar_orthogonal(n, seed, "cpu", torch.float64)
    ev = torch.logspace(0.0, -math.log10(cond), n, dtype=torch.float64)
    return ((Q * ev.unsqueeze(0)) @ Q.t()).to(dtype)
