"""Host logic of bench.py's multi-rank launch (replicas only), on CPU with gloo ranks:
the timings every rank reports reduce to their maximum, and under the reference arm only
rank 0 runs and prints."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports (10 + r, 3 - r): the maxima are (10 + world - 1, 3)
        got = bench.max_over_ranks([10.0 + rank, 3.0 - rank], world, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            assert out[r] == [10.0 + world - 1, 3.0]


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]


def test_reference_arm_other_ranks_do_nothing(capsys):
    class A:  # the fields run_reference reads
        small = True
        warmup = 0
        steps = 1
        gpus = 2
    bench.run_reference(A(), rank=1)
    assert capsys.readouterr().out == ""
