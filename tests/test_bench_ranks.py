"""bench.py host logic: whole-job figures over replica ranks (gloo on CPU),
and the hash naming the build an ncu capture was taken on.

A multi-GPU run is replicas only: each rank runs the same step on its own
requests and nothing crosses ranks on the data path.  The job's time is the
slowest rank's and its units are every rank's together; these tests run the
reduction bench.py uses in two processes with unequal times and units.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = [0.75, 1.25, 0.5][rank]
        units = [690.0, 552.0, 17.0][rank]
        q.put((rank, bench.job_totals(seconds, units, world)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_job_totals_take_slowest_rank_and_all_units(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = (max([0.75, 1.25, 0.5][:world]), sum([690.0, 552.0, 17.0][:world]))
    assert all(v == want for v in got.values()), got


def test_job_totals_single_rank_is_identity():
    assert bench.job_totals(0.3, 42.0, 1) == (0.3, 42.0)


def test_kernel_hash_ignores_comments_and_blank_lines():
    """The hash that names the build an ncu capture was taken on changes with
    the code, not with its comments (string literals count as code)."""
    a = 'int f() {  // one\n  return 1; /* two\n three */\n\n}\nconst char* s = "x // y";\n'
    b = 'int f() {\n  return 1;\n}\nconst char* s = "x // y";  // other words\n'
    c = 'int f() {\n  return 2;\n}\nconst char* s = "x // y";\n'
    d = 'int f() {\n  return 1;\n}\nconst char* s = "x // z";\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert bench.code_only(a) != bench.code_only(d)
    assert len(bench.kernel_source_sha()) == 16
