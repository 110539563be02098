"""The multi-process path of bench.py on the CPU (gloo, world size 2): each rank takes its own
rotation of the chunks, the step time reported is the slowest rank's, and no rank needs a GPU
for either.  The data path has no collective (replicas), so this host logic is all there is to
the N > 1 path besides the per-rank GPU work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
import bench
rank, world, _ = bench.dist_env()
dist.init_process_group("gloo")
chunks = bench.rank_rotation(["c0", "c1", "c2"], rank)
slow = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
alone = bench.max_over_ranks(3.5)
dist.barrier()
dist.destroy_process_group()
print(json.dumps(dict(rank=rank, world=world, chunks=chunks, slow=slow, alone=alone)))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_rotate_chunks_and_take_the_slowest_time():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), REPO_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    assert [o["world"] for o in outs] == [2, 2]
    assert outs[0]["chunks"] == ["c0", "c1", "c2"] and outs[1]["chunks"] == ["c1", "c2", "c0"]
    assert [o["slow"] for o in outs] == [15.0, 15.0]     # max over ranks, seen by both
    assert [o["alone"] for o in outs] == [3.5, 3.5]      # no process group: the value itself


def test_rank_rotation_covers_every_chunk_once():
    sys.path.insert(0, ROOT)
    import bench
    for n in (1, 3, 4):
        items = list(range(n))
        for r in range(6):
            rot = bench.rank_rotation(items, r)
            assert sorted(rot) == items and rot[0] == r % n
