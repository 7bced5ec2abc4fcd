"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing and whole-job aggregation, and the reference arm's
rank > 0 early exit.  The decode path itself has no collective."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [0.5, 2.0][rank]
    dt, value = bench.combine_ranks(local, step_bytes=1e9, steps=10, world=world)
    q.put((rank, dt, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, dt, value in res:
        assert dt == 2.0                      # the slowest rank sets the time
        assert value == pytest.approx(2 * 1e9 * 10 / 2.0 / 1e9)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dt, value = bench.combine_ranks(0.25, step_bytes=2e9, steps=5, world=1)
    assert dt == 0.25 and value == pytest.approx(40.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_step_sample", lambda *a, **k: called.append(1))
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert called == []
