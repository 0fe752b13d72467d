"""Benchmark of the GIFT gradient codec (libgift) on the 600M-like selective workload.

One step = one pass of the codec over one batch of synthetic gradients of the
Llama-600M-like selective deployment: 13 fc2 layers (1536 x 6144) take the
geometry-aware branch (rank-32 input-side whitening, E4M3 per-tensor local scale)
and 60 Euclidean tensors (1536 x 1536 / 1536 x 6144) take the Euclidean path
(AllReduceMax'd shared scale), each over R = 8 replica gradients held in HBM:
  geometry-aware layer: 8 x gift_encode -> gift_replica_reduce -> gift_decode
  Euclidean tensor:     8 x (amax -> shared amax -> gift_encode with it) -> gift_replica_reduce
                        (the first two steps are one gift_encode_replicas_shared call)
The factor refresh (gift_factor_update on each layer's activations, T = 16384 BF16)
runs every K = 50 steps in the method and is timed separately.

value = FP32 gradient bytes entering the codec per step (sum over tensors of
R * 4 * d_out * d_in) / step time, in GB/s, device-resident inputs, inputs larger
than L2 (so no flush is needed).  Each stage group is captured in its own CUDA graph;
a step replays the five graphs on one stream and CUDA events between them give each
group's time inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gift|reference]
With N > 1 (under torch.distributed.run) every rank runs the same per-GPU workload
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GIFT encode+decode GB/s of FP32 gradient and % HBM roofline, 600M-like fc2"
UNIT = "GB/s"
FMT = "e4m3"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="gift", choices=["gift", "reference"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-configs", action="store_true", help="skip the other configurations' measurements")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layers", type=int, default=13, help="geometry-aware layers (13 in the workload)")
    p.add_argument("--euclid", type=int, default=30, help="Euclidean tensors of each shape (30 in the workload)")
    p.add_argument("--streams", type=int, default=4, help="streams the independent tensors of a stage spread over")
    return p.parse_args()


def dist_info():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(world, backend):
    """One process per GPU (torch.distributed.run sets RANK / WORLD_SIZE / MASTER_*)."""
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)


def max_over_ranks(x, world, device):
    """The slowest rank's time: the job is done when every rank is."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, bytes_per_rank, ms):
    """Whole-job throughput in GB/s: every rank codes its own replicas (weak scaling)."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def fidelity_stats(g_hat, g):
    """RelL2, Cos, MaxErr and MSE of a decoded gradient against the FP32 mean of the replica
    gradients, in float64 (the fidelity measures of the GIFT reading notes, simplification 1,
    eq. (15))."""
    import torch
    gh = g_hat.double().reshape(-1)
    gg = g.double().reshape(-1)
    e = gh - gg
    ng, nh = torch.linalg.norm(gg), torch.linalg.norm(gh)
    fin = lambda x: float(x) if math.isfinite(float(x)) else None   # noqa: E731  (strict JSON)
    return {"rel_l2": fin(torch.linalg.norm(e) / ng), "cos": fin(torch.dot(gh, gg) / (nh * ng)),
            "max_err": fin(e.abs().max()), "mse": fin(torch.dot(e, e) / e.numel())}


def solo_call_ms(graph, calls, reps):
    """Average duration of one call when the calls of a captured graph run back to back."""
    import torch
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(max(1, reps)):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / max(1, reps) / calls


# stage group -> (ncu summary under profiles/, the kernel source its counters belong to)
PROFILES = {"gift_encode": ("encode_batch_1536x6144.md", "lowrank_batch.cu"),
            "euclid_encode": ("encode_shared_600m_shapes.md", "quant.cu")}


def profiled_traffic(group):
    """DRAM bytes per call of the group from the committed ncu summary, or None when the
    kernel source has changed since the counters were taken."""
    import hashlib
    import re
    if group not in PROFILES:
        return None
    name, source = PROFILES[group]
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(group + r"_traffic_bytes_per_call:\s*([0-9]+)", text)
    src = os.path.join(ROOT, "fac_whitening_gb300", "csrc", source)
    if not (m_src and m_b and os.path.exists(src)):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m_src.group(1):
        return None
    return int(m_b.group(1))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# --------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# --------------------------------------------------------------------------------------
def oracle_sample_step(sample, O):
    """One codec pass of the sample through the oracle statement O (oracle.cpp or numpy)."""
    W_g, W_e, F = sample["gift"], sample["euclid"], sample["factor"]
    xf = O.Xform("lowrank", F=F)
    qs = [O.encode_layer(W, xf, FMT)[0] for W in W_g]
    X = O.replica_reduce(qs, FMT)
    O.decode_layer(X, xf)
    shared = max(O.abs_max(W) for W in W_e)
    qe = [O.quantize(W, FMT, amax=shared) for W in W_e]
    O.replica_reduce(qe, FMT)


def make_oracle_sample(rows, R=8):
    """One geometry-aware layer and one Euclidean tensor, `rows` x 6144, R replicas (CPU)."""
    import torch
    import oracle.cpp as OC
    from fac_whitening_gb300 import synth
    spec = synth.LayerSpec("sample", rows, 6144, T=2048, exponent=1.0)
    Ws, a = synth.layer_inputs(spec, 2, 77, R, device="cpu")
    F = OC.lowrank_factor_from_activations(a.to(torch.float64).numpy(), r=32, iters=8)
    We = [synth.gaussian((rows, 6144), synth.seed_for(2, 99, r)).numpy() for r in range(R)]
    nbytes = 2 * R * rows * 6144 * 4
    return {"gift": [W.numpy() for W in Ws], "euclid": We, "factor": F, "bytes": nbytes,
            "desc": f"one 600M-like fc2 layer ({rows}x6144 rows of 1536x6144, rank 32) and one Euclidean "
                    f"{rows}x6144 tensor, R={R}: encode, reduce, decode"}


def cpu_cores():
    return os.cpu_count() or 1


def time_oracle(sample, steps, warmup=0, openmp=False):
    """Seconds per step of the C++ oracle: single-threaded and pinned to one host core
    (taskset -c <core>), or the OpenMP build of the same source on every core this process may
    use.  Returns (seconds, threads)."""
    import oracle.cpp as OC
    allowed = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    threads = OC.use_openmp(openmp)
    try:
        if not openmp and allowed:
            os.sched_setaffinity(0, {min(allowed)})
        for _ in range(warmup):
            oracle_sample_step(sample, OC)
        t0 = time.perf_counter()
        for _ in range(steps):
            oracle_sample_step(sample, OC)
        dt = (time.perf_counter() - t0) / max(steps, 1)
    finally:
        if allowed:
            os.sched_setaffinity(0, allowed)
        OC.use_openmp(False)
    return dt, threads


def cpu_baseline_entry(sample, dt, threads, omp=None):
    e = {"value": sample["bytes"] / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
         "sample": sample["desc"], "seconds": dt,
         "oracle": "plain C++17 (oracle/gift_oracle.cpp), -O2 -ffp-contract=off, one thread pinned to one core"}
    if omp is not None:
        odt, othreads = omp
        e["all_cores"] = {"value": sample["bytes"] / odt / 1e9, "unit": UNIT, "cores": othreads, "seconds": odt,
                          "oracle": "the same source built with OpenMP"}
    return e


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    # each step is a bounded sample, so that --steps K --warmup W ends within a few minutes
    sample = make_oracle_sample(rows=512)   # about 2 s per step on one core
    dt, threads = time_oracle(sample, args.steps, args.warmup)
    value = sample["bytes"] / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 transform, f32 quantiser", "data": "synthetic",
            "config": {"workload": "llama600m-selective (oracle sample)", "sample": sample["desc"]},
            "cpu_baseline": cpu_baseline_entry(sample, dt, threads),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, index):
        self.proc = None
        self.index = index
        # raw samples (the JSON line carries their summary); GIFT_BENCH_CLOCKS_DIR keeps them
        out_dir = os.environ.get("GIFT_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"gift_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        import shutil
        if shutil.which("nvidia-smi") is None:   # nothing to sample on this machine
            return self
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sms)}


def build_workload(args, dev):
    import torch
    from fac_whitening_gb300 import synth
    wl = synth.llama600m_selective_workload(seed_layers=args.layers, euclid_each=args.euclid)
    R = wl.R
    gift_layers, euclid = [], []
    for li, spec in enumerate(wl.layers):
        if spec.kind == "gift":
            Ws, a = synth.layer_inputs(spec, wl.config, li, R, device=dev)
            gift_layers.append({"spec": spec, "W": Ws, "a": a})
        else:
            Ws, _ = synth.layer_inputs(spec, wl.config, li, R, device=dev)
            euclid.append({"spec": spec, "W": Ws})
    torch.cuda.synchronize()
    return wl, gift_layers, euclid


def main_gift(args):
    import numpy as np
    import torch

    from fac_whitening_gb300 import gift as G

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    ctx = G.Context(local)
    hbm_peak, bf16_peak, peak_kind = peaks()

    wl, gl, eu = build_workload(args, dev)
    R = wl.R
    stream = torch.cuda.current_stream()
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    # ---- factor refresh (timed separately) -------------------------------------------
    d_out, d_in = 1536, 6144
    T = gl[0]["a"].shape[0] if gl else 0
    fws = torch.zeros(G.gift_workspace_bytes(ctx, "factor_update", "lowrank", FMT, "tensor", d_out, d_in, T),
                      dtype=torch.uint8, device=dev)
    factors = []
    fe0, fe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i, L in enumerate(gl):   # the codec's factors carry their U term planes (refreshed with U)
        f = G.Factor.empty("lowrank", d_out, d_in, 32, device=dev, planes=True)
        factors.append(f)
    # the codec uses the FP32-precision factors; the tensor-core (TC precision) refresh is
    # timed beside it on the same activations
    refresh = {}
    replayed = True
    for prec in ("tc", "fp32"):
        if not gl:
            break
        scratch = [G.Factor.empty("lowrank", d_out, d_in, 32, device=dev) for _ in gl] if prec == "tc" else factors
        G.gift_factor_update(ctx, scratch[0], gl[0]["a"], seed=1, prec=prec, ws=fws, status=st)   # warm-up
        torch.cuda.synchronize()

        def refresh_seq(scratch=scratch, prec=prec):
            for i, L in enumerate(gl):
                G.gift_factor_update(ctx, scratch[i], L["a"], seed=1000 + i, prec=prec, ws=fws, status=st)

        ms, rep = graph_ms(refresh_seq)
        replayed = replayed and rep
        refresh[prec] = ms / len(gl)
    factor_ms = refresh.get("fp32", 0.0)
    # all the layers refreshed together, as Algorithm 1 refreshes them every K steps: eight at a
    # time on side streams, each with its own workspace.  The refresh's 64 x 64 steps are
    # single-CTA dependent chains and its sketches fill the GPU; the layers' chains overlap the
    # other layers' sketches (measured: 1, 2, 4, 8, 13 streams gave 5.67, 4.02, 3.27, 2.87,
    # 2.88 ms per layer; quarter-GPU contexts did worse).  Scratch factors: the codec keeps
    # the factors refreshed above.
    if gl:
        nrs = 8
        rws = [torch.zeros(fws.numel(), dtype=torch.uint8, device=dev) for _ in range(nrs)]
        rstreams = [torch.cuda.Stream() for _ in range(nrs)]
        rscratch = [G.Factor.empty("lowrank", d_out, d_in, 32, device=dev) for _ in gl]

        def refresh_all():
            main = torch.cuda.current_stream()
            for s_ in rstreams:
                s_.wait_stream(main)
            for i, L in enumerate(gl):
                j = i % nrs
                with torch.cuda.stream(rstreams[j]):
                    G.gift_factor_update(ctx, rscratch[i], L["a"], seed=1000 + i, prec="fp32", ws=rws[j], status=st)
            for s_ in rstreams:
                main.wait_stream(s_)

        refresh_all()
        torch.cuda.synchronize()
        ms, rep = graph_ms(refresh_all)
        replayed = replayed and rep
        refresh["fp32_all_layers"] = ms / len(gl)
        del rws, rscratch
        torch.cuda.empty_cache()
    # the K-FAC factor alone on the tensor cores (gift_kfac_factor: transpose, tcgen05 SYRK of
    # the lower tiles, mirror), d (d + 1) T flops
    kfac = None
    if gl:
        Abuf = torch.empty(d_in, d_in, device=dev)
        kws = torch.zeros(G.gift_workspace_bytes(ctx, "kfac_factor", "identity", FMT, "tensor", d_in, d_in, T),
                          dtype=torch.uint8, device=dev)
        G.gift_kfac_factor(ctx, gl[0]["a"], Abuf, prec="tc", ws=kws, status=st)
        torch.cuda.synchronize()
        fe0.record()
        for _ in range(5):
            G.gift_kfac_factor(ctx, gl[0]["a"], Abuf, prec="tc", ws=kws, status=st)
        fe1.record()
        torch.cuda.synchronize()
        kms = fe0.elapsed_time(fe1) / 5
        kflops = float(d_in) * (d_in + 1) * T
        kfac = {"ms": kms, "tflops": kflops / (kms * 1e-3) / 1e12, "peak_tflops": bf16_peak,
                "frac": kflops / (kms * 1e-3) / 1e12 / bf16_peak, "peak_kind": peak_kind + " bf16 burst",
                "flops": kflops, "shape": f"a {T}x{d_in} BF16 -> A {d_in}x{d_in} FP32"}
        del Abuf, kws
    for L in gl:
        del L["a"]
    torch.cuda.empty_cache()

    # ---- buffers -----------------------------------------------------------------------
    ws_bytes = max(G.gift_workspace_bytes(ctx, op, k, FMT, "tensor", d_out, d_in)
                   for op in ("encode", "decode", "amax") for k in ("lowrank", "identity"))
    nstr = max(1, args.streams)
    streams = [torch.cuda.Stream() for _ in range(nstr)]
    wss = [torch.zeros(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(nstr)]

    def codes_for(spec):
        return ([torch.empty(spec.d_out * spec.d_in, dtype=torch.uint8, device=dev) for _ in range(R)],
                [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(R)])

    for L in gl:
        L["codes"], L["scales"] = codes_for(L["spec"])
        L["avg"] = torch.empty(d_out, d_in, dtype=torch.float32, device=dev)
        L["out"] = torch.empty(d_out, d_in, dtype=torch.float32, device=dev)
    shared = torch.zeros(max(len(eu), 1), dtype=torch.float32, device=dev)
    for j, E in enumerate(eu):
        E["codes"], E["scales"] = codes_for(E["spec"])
        E["avg"] = torch.empty(E["spec"].d_out, E["spec"].d_in, dtype=torch.float32, device=dev)
        E["shared"] = shared[j:j + 1]

    solo_mode = [False]

    # The layers' decodes are latency-bound one by one: they run side by side, each stream's
    # context sized for its share of the SMs (GIFT_OPT_SMS), with workspaces sized by it.
    ctx_q = G.Context(local)
    G.gift_set_option(ctx_q, G.OPT_SMS, max(1, torch.cuda.get_device_properties(dev).multi_processor_count // nstr))
    wsq = [torch.zeros(max(G.gift_workspace_bytes(ctx_q, "decode", "lowrank", FMT, "tensor", d_out, d_in), 256),
                       dtype=torch.uint8, device=dev) for _ in range(nstr)]

    def fork_join(items, fn, ws_list=None):
        """Run fn(item, ws) for independent items round-robin over the side streams; the
        current stream waits for all of them (one join per stage group).  In solo mode the
        items run back to back on the current stream (per-call timing)."""
        ws_list = wss if ws_list is None else ws_list
        if solo_mode[0]:
            for it in items:
                fn(it, ws_list[0])
            return
        main = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)
        for s in streams:
            s.wait_stream(main)
        for i, it in enumerate(items):
            with torch.cuda.stream(streams[i % nstr]):
                fn(it, ws_list[i % nstr])
        for s in streams:
            main.wait_stream(s)

    # ---- stage groups ------------------------------------------------------------------
    def encode_layer(f, L, w, stream=None):
        # the layer's R replicas in one call (one cooperative launch)
        G.gift_encode_replicas(ctx, f, L["W"], FMT, "tensor", L["codes"], scales=L["scales"], ws=w, status=st,
                               stream=stream)

    def g_encode():
        fork_join(list(zip(factors, gl)), lambda it, w: encode_layer(it[0], it[1], w))

    def g_reduce():
        fork_join(gl, lambda L, w: G.gift_replica_reduce(ctx, L["codes"], L["scales"], FMT, "tensor", d_out, d_in,
                                                         L["avg"], status=st))

    def g_decode():
        fork_join(list(zip(factors, gl)),
                  lambda it, w: G.gift_decode(ctx_q, it[0], it[1]["avg"], False, "f32", "tensor", d_out, d_in,
                                              it[1]["out"], ws=w, status=st), ws_list=wsq)

    def euclid_encode(E, w):
        # the R replicas' shared amax and their pack with it: one cooperative launch
        G.gift_encode_replicas_shared(ctx, None, E["W"], FMT, "tensor", E["codes"], E["scales"],
                                      shared_amax_out=E["shared"], ws=w, status=st)

    def e_encode():
        fork_join(eu, euclid_encode)

    def e_reduce():
        fork_join(eu, lambda E, w: G.gift_replica_reduce(ctx, E["codes"], E["scales"], FMT, "tensor",
                                                         E["spec"].d_out, E["spec"].d_in, E["avg"], status=st))

    groups = [("gift_encode", g_encode), ("gift_reduce", g_reduce), ("gift_decode", g_decode),
              ("euclid_encode", e_encode), ("euclid_reduce", e_reduce)]
    n_gift = len(gl) * d_out * d_in
    n_eu = sum(E["spec"].d_out * E["spec"].d_in for E in eu)
    # algorithmic bytes and launches of each group (per step)
    # (gift_encode_replicas: projection pass, Pc reduce, apply-and-pack pass; the decode of a
    # factor with cached planes: tensor-core projection and the pipelined apply)
    alg = {"gift_encode": (R * n_gift * 5, len(gl) * 3, len(gl)),
           "gift_reduce": (n_gift * (R + 4), len(gl), len(gl)),
           "gift_decode": (n_gift * 8, len(gl) * 2, len(gl)),
           "euclid_encode": (R * n_eu * 5, len(eu), len(eu)),
           "euclid_reduce": (n_eu * (R + 4), len(eu), len(eu))}
    kernels_per_step = sum(v[1] for v in alg.values())
    grad_bytes = R * 4 * (n_gift + n_eu)

    # eager warm-up (also loads every kernel), then capture one graph per group
    for _, fn in groups:
        fn()
    torch.cuda.synchronize()
    graphs = []
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        for name, fn in groups:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs.append((name, g))
    torch.cuda.synchronize()
    # every group's calls back to back on a single stream, for the per-call roofline timing
    graphs_solo = {}
    solo_mode[0] = True
    with torch.cuda.stream(cap):
        for name, fn in groups:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs_solo[name] = g
    solo_mode[0] = False
    torch.cuda.synchronize()

    def step(evs=None):
        for i, (name, g) in enumerate(graphs):
            g.replay()
            if evs is not None:
                evs[i + 1].record()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st.zero_()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record()
        for k in range(args.steps):
            ev[k][0].record()
            step(ev[k])
        t1.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms = total_ms / args.steps
    status_word = int(st.item())
    group_ms = {name: sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)) / args.steps
                for i, (name, _) in enumerate(graphs)}
    value = job_value(world, grad_bytes, ms)

    # ---- fidelity of one geometry-aware layer (after the timed region) -----------------
    # the decoded layer against the FP32 mean of its replicas, and the same replicas through
    # the Euclidean codec (shared scale) for comparison
    try:
        L0 = gl[0]
        gbar = torch.zeros(d_out, d_in, dtype=torch.float64, device=dev)
        for W in L0["W"]:
            gbar += W.double()
        gbar /= len(L0["W"])
        fid = {"gift": fidelity_stats(L0["out"], gbar)}
        ecodes = [torch.empty_like(c) for c in L0["codes"]]
        escales = [torch.empty_like(x) for x in L0["scales"]]
        eavg = torch.empty_like(L0["avg"])
        fst = torch.zeros(1, dtype=torch.int32, device=dev)
        G.gift_encode_replicas_shared(ctx, None, L0["W"], FMT, "tensor", ecodes, escales, ws=wss[0], status=fst)
        G.gift_replica_reduce(ctx, ecodes, escales, FMT, "tensor", d_out, d_in, eavg, status=fst)
        torch.cuda.synchronize()
        fid["euclid_same_layer"] = fidelity_stats(eavg, gbar)
        fid["device_status"] = int(fst.item())
        fid["layer"] = f"fc2.0 {d_out}x{d_in}, R={R}, {FMT} per-tensor"
        del ecodes, escales, eavg, gbar
    except Exception as ex:   # a measurement, never a reason to lose the bench line
        fid = {"error": str(ex)[:200]}

    # ---- the other configurations and the fidelity per format ---------------------------
    configs = None
    if not args.no_configs and rank == 0:
        try:
            configs = other_configs(G, ctx, dev, hbm_peak, bf16_peak, peak_kind,
                                    gl0=gl[0]["W"] if gl else None, f0=factors[0] if factors else None)
        except Exception as ex:   # a measurement, never a reason to lose the bench line
            configs = {"error": str(ex)[:200]}

    # ---- roofline of the dominant kernel ----------------------------------------------
    # The dominant group is the Euclidean shared-scale encode (one cooperative launch per
    # tensor: amax of its R replicas, grid barrier, pack) or the rank-r encode (one
    # gift_encode_replicas call per layer: projection pass, Pc reduce, apply-and-pack pass).
    # Its call duration is timed on its own: the group's calls replayed back to back on one
    # stream (CUDA events around the replays), so calls do not overlap.
    dom = max(group_ms, key=group_ms.get)
    bytes_g, launches_g, calls_g = alg[dom]
    solo = solo_call_ms(graphs_solo.get(dom), calls_g, args.steps) if graphs_solo.get(dom) else None
    per_call_ms = solo if solo else group_ms[dom] / calls_g
    achieved = bytes_g / calls_g / (per_call_ms * 1e-3) / 1e9
    traffic = profiled_traffic(dom)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "kernel": dom,
                "peak_kind": peak_kind, "per_call_us": per_call_ms * 1e3,
                "per_call_timing": "back-to-back on one stream" if solo else "group time / calls",
                "per_call_us_in_step": group_ms[dom] / calls_g * 1e3,
                "algorithmic_bytes_per_call": bytes_g / calls_g}
    stages = {name: {"ms": group_ms[name], "share": group_ms[name] / sum(group_ms.values()),
                     "GB/s_algorithmic": alg[name][0] / (group_ms[name] * 1e-3) / 1e9,
                     "hbm_frac": alg[name][0] / (group_ms[name] * 1e-3) / 1e9 / hbm_peak}
              for name in group_ms}

    # ---- end to end through the public API with host buffers --------------------------
    e2e = None
    if not args.no_e2e:
        def item_ops(it):
            kind, i, X = it
            w = wss[0]
            if kind == "gift":
                f = factors[i]
                encode_layer(f, X, w)
                G.gift_replica_reduce(ctx, X["codes"], X["scales"], FMT, "tensor", d_out, d_in, X["avg"], status=st)
                G.gift_decode(ctx, f, X["avg"], False, "f32", "tensor", d_out, d_in, X["out"], ws=w, status=st)
            else:
                euclid_encode(X, w)
                G.gift_replica_reduce(ctx, X["codes"], X["scales"], FMT, "tensor", X["spec"].d_out,
                                      X["spec"].d_in, X["avg"], status=st)

        e2e = run_e2e(args, gl, eu, dev, grad_bytes, world, item_ops)

    # ---- CPU baseline (oracle on a bounded sample) --------------------------------------
    cpu = None
    if not args.no_cpu_baseline and rank == 0:
        sample = make_oracle_sample(rows=1536)   # the whole layer: about 7 s of single-core work
        dt, threads = time_oracle(sample, 1)
        cpu = cpu_baseline_entry(sample, dt, threads, omp=time_oracle(sample, 1, warmup=1, openmp=True))

    if rank == 0:
        clocks = clk.summary()
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32 transform, e4m3 codes", "data": "synthetic",
                "config": {"workload": "llama600m-selective: 13 fc2 1536x6144 rank-32 GIFT + 60 Euclidean "
                                       "(30x 1536x1536, 30x 1536x6144), E4M3 per-tensor, R=8",
                           "gift_layers": len(gl), "euclid_tensors": len(eu), "replicas": R,
                           "gradient_bytes_per_step": grad_bytes, "l2": "inputs exceed L2 (no flush)",
                           "parallelism": f"replicas x{world}", "streams_per_stage": nstr},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": kernels_per_step * args.steps, "stages": stages, "fidelity": fid,
                "factor_syrk": kfac, "configs": configs,
                "factor_refresh": {p: {"ms_per_layer": ms_} for p, ms_ in refresh.items()} | {
                                   "note": "whole rank-32 refresh per layer (13 layers, d_in 6144, T 16384 BF16 "
                                           "activations, CUDA events): the implicit sketch a^T (a Q) / T on the "
                                           "tensor cores, CholQR2 and Rayleigh-Ritz in FP32, stopped once the Ritz "
                                           "residuals converge (at most 16 iterations); fp32 = three-term operand "
                                           "splits (the factors the codec uses), tc = two-term, one layer after "
                                           "the other on the whole GPU; fp32_all_layers = the 13 layers refreshed "
                                           "together, eight at a time on side streams (total / 13); each sequence "
                                           "captured once into a CUDA graph and replayed (the refresh is a fixed "
                                           "launch sequence)",
                                   "graph_replay": replayed},
                "device_status": status_word}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------------------------------
# The other configurations and the fidelity per format (after the timed region)
# --------------------------------------------------------------------------------------
def graph_ms(fn):
    """(ms, replayed): one run of fn timed with CUDA events, fn's launches captured once into
    a CUDA graph and the graph replayed after one untimed replay (the host's per-launch cost
    and the gaps between launches are not in the number); eager if the capture fails."""
    import torch
    run, replayed = fn, False
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        run, replayed = g.replay, True
    except Exception:   # a call that cannot be captured: time it eagerly
        torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    run()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b), replayed


def time_cold(fn, reps=5):
    """Mean ms of fn() over reps, each run after a 256 MB write (L2 flushed), CUDA events on
    the current stream.  fn's launches are captured once into a CUDA graph and the graph is
    replayed, as the codec step replays its groups (so the host's per-call cost is not in
    the number); if the capture fails, fn runs eagerly."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    fn()
    torch.cuda.synchronize()
    run = fn
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        run = g.replay
    except Exception:   # a call that cannot be captured: time it eagerly
        torch.cuda.synchronize()
    tot = 0.0
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        tot += a.elapsed_time(b)
    return tot / reps


def codec_pass(G, ctx, f, Ws, fmt, scaling, ws_enc, ws_dec, st, prec="fp32"):
    """Buffers and closures for one layer's encode (its R replicas), reduce and decode."""
    import torch
    d_out, d_in = Ws[0].shape
    R = len(Ws)
    cb, sc = G.gift_code_sizes(fmt, scaling, d_out, d_in)
    codes = [torch.empty(cb, dtype=torch.uint8, device="cuda") for _ in range(R)]
    sdt = torch.uint8 if fmt == "nvfp4" else torch.float32
    scales = [torch.empty(sc, dtype=sdt, device="cuda") for _ in range(R)]
    tsc = [torch.empty(1, device="cuda") for _ in range(R)] if fmt == "nvfp4" else None
    avg = torch.empty(d_out, d_in, device="cuda")
    out = torch.empty(d_out, d_in, device="cuda")
    P = {"codes": codes, "scales": scales, "tsc": tsc, "avg": avg, "out": out}
    P["encode"] = lambda: G.gift_encode_replicas(ctx, f, Ws, fmt, scaling, codes, scales=scales, tensor_scales=tsc,
                                                  prec=prec, ws=ws_enc, status=st)
    P["reduce"] = lambda: G.gift_replica_reduce(ctx, codes, scales, fmt, scaling, d_out, d_in, avg,
                                                tensor_scales=tsc, status=st)
    P["decode"] = lambda: G.gift_decode(ctx, f, avg, False, "f32", "tensor", d_out, d_in, out, prec=prec,
                                        ws=ws_dec, status=st)
    return P


def measure_codec(G, ctx, f, Ws, fmt, scaling, st, hbm_peak, prec="fp32", reps=5):
    """GB/s of FP32 gradient (4 bytes per element of every replica) and the fraction of the HBM
    peak on the algorithmic bytes of each stage: encode 4 + code bytes, reduce R x code bytes
    + 4, decode 8 per element."""
    import torch
    d_out, d_in = Ws[0].shape
    kind = "identity" if f is None else f.kind
    R = len(Ws)
    n = d_out * d_in
    cbytes = {"nvfp4": 0.5 + 1 / 16, "f32": 4}.get(fmt, 1.0)
    ws_enc = torch.zeros(max(G.gift_workspace_bytes(ctx, "encode", kind, fmt, scaling, d_out, d_in), 256),
                         dtype=torch.uint8, device="cuda")
    ws_dec = torch.zeros(max(G.gift_workspace_bytes(ctx, "decode", kind, "f32", "tensor", d_out, d_in), 256),
                         dtype=torch.uint8, device="cuda")
    P = codec_pass(G, ctx, f, Ws, fmt, scaling, ws_enc, ws_dec, st, prec)
    res = {}
    alg = {"encode": R * n * (4 + cbytes), "reduce": n * (R * cbytes + 4), "decode": n * 8}
    for stage in ("encode", "reduce", "decode"):
        ms = time_cold(P[stage], reps)
        res[stage] = {"us": ms * 1e3, "GB/s_gradient": (R if stage == "encode" else 1) * 4 * n / (ms * 1e-3) / 1e9,
                      "hbm_frac": alg[stage] / (ms * 1e-3) / 1e9 / hbm_peak}
    return res, P


def fidelity_gift_vs_euclid(G, ctx, f, Ws, fmt, st):
    """RelL2, Cos, MaxErr, MSE (eq. (15)) of the decoded layer against the FP32 mean of its
    replicas: GIFT (the factor's transform, per-replica scales) and the Euclidean path (identity,
    the replicas' shared scale)."""
    import torch
    d_out, d_in = Ws[0].shape
    kind = f.kind
    gbar = torch.zeros(d_out, d_in, dtype=torch.float64, device="cuda")
    for W in Ws:
        gbar += W.double()
    gbar /= len(Ws)
    ws_enc = torch.zeros(G.gift_workspace_bytes(ctx, "encode", kind, fmt, "tensor", d_out, d_in),
                         dtype=torch.uint8, device="cuda")
    ws_dec = torch.zeros(G.gift_workspace_bytes(ctx, "decode", kind, "f32", "tensor", d_out, d_in),
                         dtype=torch.uint8, device="cuda")
    P = codec_pass(G, ctx, f, Ws, fmt, "tensor", ws_enc, ws_dec, st)
    P["encode"]()
    P["reduce"]()
    P["decode"]()
    E = codec_pass(G, ctx, None, Ws, fmt, "tensor", ws_enc, ws_dec, st)
    G.gift_encode_replicas_shared(ctx, None, Ws, fmt, "tensor", E["codes"], E["scales"], tensor_scales=E["tsc"],
                                  ws=ws_enc, status=st)
    E["reduce"]()
    torch.cuda.synchronize()
    return {"gift": fidelity_stats(P["out"], gbar), "euclid": fidelity_stats(E["avg"], gbar)}


def other_configs(G, ctx, dev, hbm_peak, bf16_peak, peak_kind, gl0=None, f0=None):
    """One line per configuration besides the timed 600M-like step: codec GB/s per stage and
    format, the factor refresh, and the fidelity per format, GIFT against Euclidean."""
    import torch
    from fac_whitening_gb300 import synth
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}

    def refresh_ms(kind, a, d_out, delta=None, prec="fp32"):
        d_in = a.shape[1]
        f = G.Factor.empty(kind, d_out, d_in, 32, device=dev)
        w = torch.zeros(G.gift_workspace_bytes(ctx, "factor_update", kind, FMT, "tensor", d_out, d_in, a.shape[0]),
                        dtype=torch.uint8, device=dev)
        ms = time_cold(lambda: G.gift_factor_update(ctx, f, a, delta=delta, seed=3, prec=prec, ws=w, status=st), 2)
        del w
        return f, ms

    # ---- tiny single layer: 64 x 256, T = 512 FP32, rank 32, E4M3, R = 4 -----------------
    try:
        wl = synth.tiny_workload()
        spec = wl.layers[0]
        Ws, a = synth.layer_inputs(spec, wl.config, 0, wl.R, device=dev)
        f, fms = refresh_ms("lowrank", a, spec.d_out)
        codec, _ = measure_codec(G, ctx, f, Ws, "e4m3", "tensor", st, hbm_peak)
        out["tiny_64x256"] = {"factor_refresh_ms": fms, "codec_e4m3": codec,
                              "fidelity_e4m3": fidelity_gift_vs_euclid(G, ctx, f, Ws, "e4m3", st)}
    except Exception as ex:
        out["tiny_64x256"] = {"error": str(ex)[:200]}

    # ---- 300M-like fc2: 1024 x 4096, T = 8192 BF16, R = 8; every transform --------------
    try:
        wl = synth.llama300m_fc2_workload()
        spec = wl.layers[0]
        Ws, a = synth.layer_inputs(spec, wl.config, 0, wl.R, device=dev)
        delta = synth.delta_for_layer(spec, wl.config, 0, device=dev)
        res = {}
        for kind in ("chol_two_sided", "chol_input", "lowrank"):
            f, fms = refresh_ms(kind, a, spec.d_out, delta=delta if kind == "chol_two_sided" else None)
            codec, _ = measure_codec(G, ctx, f, Ws, "e4m3", "tensor", st, hbm_peak)
            entry = {"factor_refresh_ms": fms, "codec_e4m3": codec,
                     "fidelity_e4m3": fidelity_gift_vs_euclid(G, ctx, f, Ws, "e4m3", st)}
            if kind != "lowrank":   # triangular products W L^-T (d_in^2 d_out) and L_G^-1 X (d_out^2 d_in)
                fl = spec.d_out * spec.d_in * spec.d_in + (spec.d_out ** 2 * spec.d_in if kind == "chol_two_sided" else 0)
                entry["transform_tflops_fp32_equivalent"] = fl / (codec["encode"]["us"] * 1e-6 / wl.R) / 1e12
            res[kind] = entry
            del f
        codec, _ = measure_codec(G, ctx, None, Ws, "e4m3", "tensor", st, hbm_peak)
        res["identity"] = {"codec_e4m3": codec}
        out["llama300m_fc2_1024x4096"] = res
        del Ws, a, delta
    except Exception as ex:
        out["llama300m_fc2_1024x4096"] = {"error": str(ex)[:200]}
    torch.cuda.empty_cache()

    # ---- 600M-like fc2 layer 0: fidelity per format ------------------------------------
    if gl0 is not None and f0 is not None:
        try:
            out["llama600m_fc2_fidelity"] = {fmt: fidelity_gift_vs_euclid(G, ctx, f0, gl0, fmt, st)
                                             for fmt in ("e4m3", "e5m2", "nvfp4")}
            codec, _ = measure_codec(G, ctx, f0, gl0, "nvfp4", "tensor", st, hbm_peak)
            out["llama600m_fc2_codec_nvfp4"] = codec
            codec, _ = measure_codec(G, ctx, f0, gl0, "e5m2", "tensor", st, hbm_peak)
            out["llama600m_fc2_codec_e5m2"] = codec
        except Exception as ex:
            out["llama600m_fc2_fidelity"] = {"error": str(ex)[:200]}

    # ---- profiler + per-block scaling: 48 heavy-tailed gradients -----------------------
    try:
        wl = synth.profiler_workload()
        grads = [synth.layer_inputs(sp, wl.config, i, 1, device=dev)[0][0] for i, sp in enumerate(wl.layers)]
        n_all = sum(g.numel() for g in grads)
        res = {}
        counts = torch.zeros(len(grads), 3, dtype=torch.int64, device=dev)
        wsa = torch.zeros(max(G.gift_workspace_bytes(ctx, "amax", "identity", "e4m3", "tensor", 6144, 6144), 256),
                          dtype=torch.uint8, device=dev)
        for fmt in ("e4m3", "e5m2"):
            def hits():   # the 48 tensors in one call: two launches
                counts.zero_()
                G.gift_boundary_hit_rates(ctx, grads, fmt, "tensor", counts, ws=wsa, status=st)
            ms = time_cold(hits, 3)
            res[f"hit_rate_{fmt}"] = {"us_all_48": ms * 1e3, "GB/s_gradient": 4 * n_all / (ms * 1e-3) / 1e9,
                                      "hbm_frac": 4 * n_all / (ms * 1e-3) / 1e9 / hbm_peak}
        counts.zero_()   # the selection uses the E4M3 counts
        G.gift_boundary_hit_rates(ctx, grads, "e4m3", "tensor", counts, ws=wsa, status=st)
        order, _, k = G.gift_select_fragile(counts.cpu().numpy().astype("uint64"), 13)
        sel = [grads[i] for i in order[:k]]
        # the selected layers encoded with 128 x 128 block scales after a rank-32 whitening
        fac = {}
        for g in sel:
            if g.shape[1] not in fac:
                q, _ = torch.linalg.qr(torch.randn(g.shape[1], 32, device=dev))
                fac[g.shape[1]] = (q.contiguous(), torch.linspace(40, 1, 32, device=dev))
        n_sel = sum(g.numel() for g in sel)
        bufs = []
        for g in sel:
            U, mu = fac[g.shape[1]]
            f = G.Factor("lowrank", g.shape[0], g.shape[1], 32, U=U, mu=mu, sigma=torch.tensor([0.1], device=dev))
            cb, sc = G.gift_code_sizes("e4m3", "block128", *g.shape)
            w = torch.zeros(G.gift_workspace_bytes(ctx, "encode", "lowrank", "e4m3", "block128", *g.shape),
                            dtype=torch.uint8, device=dev)
            bufs.append((f, g, torch.empty(cb, dtype=torch.uint8, device=dev), torch.empty(sc, device=dev), w))

        def enc13():
            for f, g, c, s_, w in bufs:
                G.gift_encode(ctx, f, g, "e4m3", "block128", c, s_, ws=w, status=st)
        ms = time_cold(enc13, 3)
        res["top13_block128_rank32_encode"] = {"us_all_13": ms * 1e3, "GB/s_gradient": 4 * n_sel / (ms * 1e-3) / 1e9,
                                               "hbm_frac": 5 * n_sel / (ms * 1e-3) / 1e9 / hbm_peak,
                                               "selected": [int(i) for i in order[:k]]}
        out["profiler_48"] = res
        del grads, sel, bufs
    except Exception as ex:
        out["profiler_48"] = {"error": str(ex)[:200]}
    torch.cuda.empty_cache()

    # ---- large stress: one fc2-like 4096 x 16384 layer, R = 16, E4M3 and NVFP4 ----------
    try:
        D_OUT, D_IN, R = 4096, 16384, 16
        gen = torch.Generator(device=dev).manual_seed(62)
        U, _ = torch.linalg.qr(torch.randn(D_IN, 32, generator=gen, device=dev))
        mu = (1.0 / torch.arange(1, 33, device=dev, dtype=torch.float32))
        mu[torch.randperm(32, generator=torch.Generator().manual_seed(5))[:8].to(dev)] *= 100.0
        mu = torch.sort(mu, descending=True).values
        f = G.Factor("lowrank", D_OUT, D_IN, 32, U=U.contiguous(), mu=mu, sigma=torch.tensor([0.01], device=dev))
        Ws = []
        for _ in range(R):
            W = torch.randn(D_OUT, D_IN, generator=gen, device=dev) * 0.1
            W += (torch.randn(D_OUT, 32, generator=gen, device=dev) * 3.0) @ U.T
            Ws.append(W.contiguous())
        res = {}
        for fmt in ("e4m3", "nvfp4"):
            codec, P = measure_codec(G, ctx, f, Ws, fmt, "tensor", st, hbm_peak, reps=3)
            res[f"codec_{fmt}"] = codec
            del P
            res[f"fidelity_{fmt}"] = fidelity_gift_vs_euclid(G, ctx, f, Ws, fmt, st)
        # the factor refresh at this size: T = 32768 BF16 activations with the spectrum i^-1
        # and 8 spikes (coordinate eigenvectors: the sketch's convergence is the same)
        del Ws
        torch.cuda.empty_cache()
        s = synth.spectrum_power_law(D_IN, 1.0)
        s[synth.spike_indices(D_IN, 8, 5)] *= 10.0
        a = (torch.randn(32768, D_IN, generator=gen, device=dev) * s.to(dev, torch.float32)).to(torch.bfloat16)
        _, fms = refresh_ms("lowrank", a, D_OUT)
        res["factor_refresh_ms"] = fms
        out["stress_4096x16384_R16"] = res
        del a, f
    except Exception as ex:
        out["stress_4096x16384_R16"] = {"error": str(ex)[:200]}
    torch.cuda.empty_cache()
    out["device_status"] = int(st.item())
    return out


def near_gpu_cpus(device):
    """The CPU cores the platform lists as local to the GPU (sysfs, by its PCI address), or
    None.  Pinned host buffers allocated and first touched by a thread on those cores sit on
    the GPU's own memory node."""
    import torch
    p = torch.cuda.get_device_properties(device)
    dom, bus, dv = (getattr(p, "pci_domain_id", None), getattr(p, "pci_bus_id", None),
                    getattr(p, "pci_device_id", None))
    if bus is None or dom is None or dv is None:
        return None
    path = f"/sys/bus/pci/devices/{dom:04x}:{bus:02x}:{dv:02x}.0/local_cpulist"
    try:
        text = open(path).read().strip()
    except OSError:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return sorted(cpus & os.sched_getaffinity(0)) or None


def run_e2e(args, gl, eu, dev, grad_bytes, world, item_ops):
    """Same step through the public API with host buffers.  Per step, every replica gradient
    is copied from pinned host memory and every decoded / averaged result is read back to
    pinned host memory.  The transfers are pipelined with the codec: a copy stream uploads
    tensor after tensor, the compute stream runs each tensor's codec calls as soon as its
    inputs have landed, and a read-back stream downloads each result as soon as it exists.
    Every rank does this; the slowest rank's time counts."""
    import torch
    cpus = near_gpu_cpus(dev)
    if cpus:
        os.sched_setaffinity(0, cpus)
    items = [("gift", i, L) for i, L in enumerate(gl)] + [("euclid", j, E) for j, E in enumerate(eu)]
    host_in = [[torch.empty(W.shape, dtype=torch.float32, pin_memory=True) for W in it[2]["W"]] for it in items]
    for hs, it in zip(host_in, items):
        for h, W in zip(hs, it[2]["W"]):
            h.copy_(W)
    outs = [it[2]["out"] if it[0] == "gift" else it[2]["avg"] for it in items]
    host_out = [torch.empty(o.shape, dtype=torch.float32, pin_memory=True) for o in outs]
    h2d = sum(h.numel() * 4 for hs in host_in for h in hs)
    d2h = sum(h.numel() * 4 for h in host_out)
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    done = [None] * len(items)        # compute of the item in the previous step

    def one_step():
        landed = []
        for k, (hs, it) in enumerate(zip(host_in, items)):
            with torch.cuda.stream(up):
                if done[k] is not None:
                    up.wait_event(done[k])     # the previous step's codec has read the buffers
                for h, W in zip(hs, it[2]["W"]):
                    W.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(up)
                landed.append(ev)
        for k, it in enumerate(items):
            comp.wait_event(landed[k])
            item_ops(it)
            ev = torch.cuda.Event()
            ev.record(comp)
            done[k] = ev
            with torch.cuda.stream(down):
                down.wait_event(ev)
                host_out[k].copy_(outs[k], non_blocking=True)
        comp.wait_stream(down)

    one_step()
    torch.cuda.synchronize()
    steps = max(1, args.e2e_steps)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0.record()
    for _ in range(steps):
        one_step()
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / steps
    return {"value": job_value(world, grad_bytes, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipeline": "per-tensor upload, codec and read-back on three streams",
            "host_cpus": f"{len(cpus)} cores local to the GPU" if cpus else "not pinned (no locality information)"}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    main_gift(args)


if __name__ == "__main__":
    main()
