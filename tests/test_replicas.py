"""Multi-process path of bench.py on the CPU: world size 2 over gloo.

The layer has no collective on its data path (tokens are independent, so
replicas each run the whole workload). What crosses ranks is the measurement:
a barrier before and after the timed region, the max of the step time over
ranks and the sum of the tokens. These tests run that plumbing in two spawned
gloo processes, and launch `bench.py --impl reference` under torchrun with two
ranks, where rank 0 alone times the oracle and prints one line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.timeout(300)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, backend="gloo")
    bench.barrier(dist)
    step_ms = 1.0 + r  # rank 1 is the slower one
    ms = bench.max_over_ranks(dist, step_ms)
    tokens = bench.sum_over_ranks(dist, 4096.0)
    bench.barrier(dist)
    q.put((r, w, local, ms, tokens, tokens / (ms / 1e3)))
    dist.destroy_process_group()


def test_replica_measurement_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, ms, tokens, value) in enumerate(out):
        assert (rank, world, local) == (r, 2, r)
        assert ms == 2.0          # the max over ranks: the slower replica sets the time
        assert tokens == 8192.0   # every replica's tokens count
        assert value == 8192.0 / 0.002


def test_without_a_process_group_the_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1) is None
    bench.barrier(None)
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 7.0) == 7.0


def test_reference_arm_under_torchrun_with_two_ranks():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
