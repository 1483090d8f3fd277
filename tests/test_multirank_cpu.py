"""Multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU).

Every rank runs its own replica of the workload; the only cross-rank
traffic is the barrier and the max-over-ranks reduction of the timed
region.  These tests run that logic with world size 2 over gloo.
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)     # rank 1 is the slow one
    bench.barrier(world)
    value = bench.job_value(world, 1000, 4, slowest)
    out.put((rank, slowest, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]                   # both ranks see the slowest time
    assert res[0][2] == pytest.approx(2 * 1000 * 4 / 0.015)     # all ranks' units over that time


def test_reference_arm_prints_once_under_two_ranks():
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_pinned_legs_must_fit_every_rank_of_the_node():
    sys.path.insert(0, ROOT)
    import bench
    gb = 10 ** 9
    # the LLaMA-2-7B end-to-end leg pins 27 GB (bf16 grads and weights) per rank
    assert bench.pinned_leg_fits(27 * gb, 1, 200 * gb)
    assert bench.pinned_leg_fits(27 * gb, 4, 200 * gb) is True       # 140 GB with headroom
    assert bench.pinned_leg_fits(27 * gb, 8, 200 * gb) is False      # 281 GB with headroom
    assert bench.pinned_leg_fits(1, 1, None) is False                # unknown memory: not enough
    avail = bench.host_mem_available()
    assert avail is None or avail > 0
