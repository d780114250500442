"""The multi-rank host logic of bench.py on CPU: two gloo ranks
(token-sharded replicas, no data-path collective; the only exchange is the
max over ranks of the step time)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, sys
sys.path.insert(0, %r)
import torch.distributed as dist
import bench, synth
rank, world, local = bench.dist_env()
dist.init_process_group("gloo", rank=rank, world_size=world)
ms = bench.max_over_ranks(1.5 + rank, dist, "cpu")
seeds = [bench.rank_token_seed(rank, c) for c in range(4)]
x = synth.gen_tokens(2, 256, bench.rank_token_seed(rank)).tolist()
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "world": world, "local": local, "ms": ms, "seeds": seeds, "x": x}))
""" % ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_the_slowest_time_and_own_their_tokens():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE="2", LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    out = []
    for p in procs:
        so, se = p.communicate(timeout=180)
        assert p.returncode == 0, se
        out.append(json.loads(so.strip().splitlines()[-1]))
    out.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in out] == [0, 1] and all(d["world"] == 2 for d in out)
    assert all(d["ms"] == 2.5 for d in out)          # max over ranks, seen by both
    assert not set(out[0]["seeds"]) & set(out[1]["seeds"])
    assert out[0]["x"] != out[1]["x"]                # each rank holds its own tokens


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(512, 1, 0.25) == pytest.approx(512 / 0.25e-3)
    assert bench.job_throughput(512, 4, 0.25) == pytest.approx(4 * 512 / 0.25e-3)
    assert bench.rank_token_seed(0) == 10 ** 6   # rank 0 keeps the single-GPU inputs
