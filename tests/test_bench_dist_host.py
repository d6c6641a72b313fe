"""bench.py's replica plumbing on CPU: two ranks over gloo (127.0.0.1) run
dist_setup, barrier and max_over_ranks as bench.py does under torchrun, and
rank 0 alone prints the reference arm's line.  No GPU: the N > 1 path of the
bench can run nowhere else here."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_CHILD = r"""
import os, sys, types, json
sys.path.insert(0, sys.argv[1])
import bench
args = types.SimpleNamespace(impl="reference")
world, rank, local, pg = bench.dist_setup(args)
assert (world, rank) == (2, int(os.environ["RANK"]))
bench.barrier(pg)
m = bench.max_over_ranks(pg, 10.0 + 5.0 * rank)
steps = int(bench.max_over_ranks(pg, float(3 + rank)))
print(json.dumps({"rank": rank, "max": m, "steps": steps}), flush=True)
pg.destroy_process_group()
"""


@pytest.mark.timeout(120)
def test_bench_two_ranks_gloo():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=110)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    # every rank sees the maximum over ranks (the bench's timing rule)
    assert [o["max"] for o in outs] == [15.0, 15.0]
    assert [o["steps"] for o in outs] == [4, 4]


@pytest.mark.timeout(300)
def test_bench_reference_arm_rank0_only():
    """The reference arm under two ranks: rank 0 prints one JSON line with
    impl "reference"; rank 1 exits 0 without output."""
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--workload", "tiny_q4", "--steps", "3", "--warmup", "3"],
            env=env, cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=280)
        assert p.returncode == 0, err[-2000:]
        outs.append([l for l in out.splitlines() if l.startswith("{")])
    assert outs[1] == []
    line = json.loads(outs[0][-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["gops"] > 0 and line["value"] > 0
