"""The N > 1 path of bench.py on CPU: one process per rank over gloo (the
path shards by batch with no data-path collective; the only cross-rank
steps are the barrier and the max-over-ranks timing)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_info() == (ws, rank, rank)
        bench.barrier(ws)
        ms = [0.25, 0.40][rank]  # the second rank is slower
        ms_max = bench.reduce_max(ms, ws, "cpu")
        results[rank] = (ms_max, bench.whole_job_rate(ws, 1_000_000_000, ms_max))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    ws = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(ws, _free_port(), results), nprocs=ws, join=True)
        got = dict(results)
    for rank in range(ws):
        ms_max, rate = got[rank]
        assert ms_max == pytest.approx(0.40)
        assert rate == pytest.approx(2 * 1e9 / 0.40e-3 / 1e9)


def test_reference_arm_on_other_ranks_does_nothing(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    called = []
    monkeypatch.setattr(bench, "run_reference", lambda *a, **k: called.append(1))
    bench.main()
    assert not called
