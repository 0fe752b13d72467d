"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The codec path does not shard (every rank codes its own replicas, weak scaling), so the
only cross-rank work is the timing: a barrier on both sides of the timed region, the
slowest rank's time, and the whole-job value.  The reference arm under a 2-rank launch
prints one line from rank 0 and nothing from the others.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_info()
    bench.dist_init(w, "gloo")
    dist.barrier()
    ms = bench.max_over_ranks(times[r], w, "cpu")
    v = bench.job_value(w, 1e9, ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, local, ms, v))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [3.5, 7.25]
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, ms, v) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert ms == 7.25                       # both ranks see the slowest rank's time
        assert v == pytest.approx(2 * 1e9 / 7.25e-3 / 1e9)   # whole-job bytes over that time


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(4.0, 1, "cpu") == 4.0
    assert bench.job_value(1, 2e9, 1000.0) == pytest.approx(2.0)
    bench.dist_init(1, "gloo")                  # no process group for one rank


@pytest.mark.timeout(600)
def test_reference_arm_two_ranks_prints_once():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=560)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
