"""The multi-process plumbing of bench.py on CPU: two gloo ranks (no GPU).

Checks the barrier, the max-over-ranks reduction of the timed region, that each
replica hashes its own batch, and that the reference arm prints on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    r, w, local = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, 1.0 + r)  # rank 1 was slower
    seed = bench.rank_seed(100, r)
    q.put((r, t, seed))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_rank_reduction_and_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [2.0, 2.0]  # both ranks see the max
    assert got[0][2] != got[1][2]  # replicas use different id batches


@pytest.mark.timeout(600)
def test_reference_arm_prints_on_rank0_only(tmp_path):
    env = dict(os.environ)
    out = []
    for rank in (0, 1):
        env.update({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank)})
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                            "--steps", "3", "--warmup", "1", "--cfg", "1"], env=env, capture_output=True, text=True,
                           timeout=600, cwd=ROOT)
        assert r.returncode == 0, r.stderr
        out.append(r.stdout.strip())
    assert out[1] == ""
    line = json.loads(out[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
