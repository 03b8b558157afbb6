"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

bench.py shards independent problems over ranks (weak scaling, no collective
on the data path).  What crosses ranks is host-side only: a barrier, the max
of the timed region and the sum of the work, and rank 0 alone printing the
JSON line.  These run here with world_size 2 on the gloo backend.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    # rank r timed (10 + r) ms over 3 steps and processed (r + 1) * 100 units
    total, units = bench.aggregate(dist, 10.0 + r, (r + 1) * 100.0)
    # the reference arm: rank 0 prints one line, the other ranks exit 0 quietly
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.reference_arm(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                   "--warmup", "3", "--workload", "dyn_n1024"]),
                                 r, w, bench.workloads.WORKLOADS["dyn_n1024"])
    bench.barrier(dist)
    dist.destroy_process_group()
    out[rank] = (r, w, total, units, rc, buf.getvalue())


def test_two_gloo_ranks_reduce_time_and_work():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, total, units, rc, text) in res.items():
        assert (r, w) == (rank, world)
        assert total == pytest.approx(11.0)          # max over ranks
        assert units == pytest.approx(300.0)         # sum over ranks
        assert rc == 0
    lines = [l for l in res[0][5].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert res[1][5].strip() == ""                   # rank 1 prints nothing
