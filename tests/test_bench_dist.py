"""The benchmark's multi-rank host logic on two gloo ranks (no GPU): rank setup from the torchrun
environment, the barrier, the max over ranks of a step time, the whole-job rate, and the reference arm that
only rank 0 runs. The decode path itself does not shard (replicas only), so this is all there is to the
N > 1 path besides the per-rank replica."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update({"WORLD_SIZE": str(ws), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_setup(None)
    bench.barrier(got_ws)
    mx = bench.max_over_ranks(times[rank], got_ws)
    out.put((got_rank, got_ws, dist.get_backend(), mx, bench.whole_job_rate(got_ws, 8, mx)))
    bench.barrier(got_ws)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [0.010, 0.025]  # seconds per step on each rank
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for rank, ws, backend, mx, rate in res:
        assert ws == 2 and backend == "gloo"
        assert mx == 0.025                   # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 8 / 0.025)   # units of both replicas over that time


def test_reference_arm_runs_on_rank_0_only(capsys, monkeypatch):
    """Under torchrun the reference arm's other ranks exit without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None, None, None) is None
    assert capsys.readouterr().out == ""
