"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks, as under
torchrun with --gpus 2 (weak scaling: every rank runs its own positions; the
job's time is the slowest rank's and its work is the sum over ranks)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        ms = [12.5, 20.0][rank]            # per-rank timed-region length
        tokens = [1000.0, 1000.0][rank]    # positions each rank processed
        ms_max = bench.max_over_ranks(ms, w)
        total = bench.sum_over_ranks(tokens, w)
        q.put((r, w, local, ms_max, total, total / (ms_max / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, ms_max, total, value) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert ms_max == 20.0                 # slowest rank sets the job time
        assert total == 2000.0                # work of all ranks
        assert value == pytest.approx(2000.0 / 0.020)


def test_single_rank_is_identity(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.sum_over_ranks(3.0, 1) == 3.0


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 0
    bench.run_reference(A())            # returns at once on a non-zero rank
    assert capsys.readouterr().out == ""
