"""The bench's multi-rank host logic on CPU: two gloo ranks (no GPU).

Every rank runs its own replica of the workload; the job's time is the
slowest rank's (an element-wise MAX all-reduce) and the reported value is the
whole job's throughput, units of all ranks over that time.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r"""
import json, os, sys
sys.path.insert(0, os.getcwd())
import torch.distributed as dist
import bench
world, rank, local = bench.dist_env()
dist.init_process_group("gloo", rank=rank, world_size=world)
vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0])
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "local": local, "max": vals}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_gloo_two_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["world"] == 2 and o["local"] == o["rank"]
        assert o["max"] == [2.0, 10.0, 5.0]  # the slowest rank per entry, on every rank


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]


def test_whole_job_rate_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    # Each of 4 ranks does 2e12 FLOP; the slowest took 0.5 s: 16e12 FLOP/s for the job.
    assert bench.whole_job_rate(2e12, 4, 0.5) == 16e12
    assert bench.whole_job_rate(2e12, 1, 0.5) == 4e12
