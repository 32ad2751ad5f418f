"""The multi-rank path of bench.py on CPU: two gloo ranks, as torchrun would start them.

bench.py runs one independent replica per GPU (no data-path collective); the only cross-rank steps are
the barrier around the timed region and the max over ranks of the measured time, from which the
whole-job rate is computed.  These run here with the gloo backend and a different "measured" time
on each rank.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
dist.barrier()
seconds = 0.5 + rank            # rank 1 is the slow replica
t = bench.max_over_ranks(seconds)
rate = bench.job_throughput(1000.0, world, 10, t)
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "t": t, "rate": rate}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("a gloo rank did not finish")
        assert p.returncode == 0, err
        outs.append(out.strip().splitlines()[-1])
    import json
    res = [json.loads(o) for o in outs]
    for r in res:
        assert r["world"] == 2
        assert r["t"] == 1.5                       # both ranks see the slowest rank's time
        assert r["rate"] == pytest.approx(1000.0 * 2 * 10 / 1.5)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_throughput(3.0, 1, 4, 2.0) == 6.0
