"""The N > 1 bench path on CPU: two gloo ranks, replicas only (no data-path collective).

Each rank times its own batch; the job's time is the slowest rank's (element-wise max over
ranks), and the job's rate counts every rank's units (weak scaling). Run as two spawned
processes on 127.0.0.1 with the gloo backend.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "measured" (10 + r) ms for the steps, (20 - r) ms end to end, 5 ms kernel
        ms, e_ms, k_ms = bench.max_over_ranks([10.0 + rank, 20.0 - rank, 5.0], world)
        out[rank] = (ms, e_ms, k_ms, bench.whole_job_rate(world, 64, ms, 4))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_units():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        ms, e_ms, k_ms, rate = res[r]
        assert ms == 11.0 and e_ms == 20.0 and k_ms == 5.0  # max over ranks, element-wise
        assert rate == pytest.approx(2 * 64 / (11.0e-3 / 4))  # both ranks' queries over the slowest time


def test_single_rank_is_the_identity():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.whole_job_rate(1, 64, 8.0, 2) == pytest.approx(64 / 4e-3)
