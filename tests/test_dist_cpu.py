"""The multi-rank bookkeeping of bench.py (max-over-ranks timing, whole-job throughput, rank-0-only
reference arm), run as world_size-2 gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank               # rank 1 is the straggler
    m = bench.reduce_max(local_ms, "cpu")
    v = bench.tokens_per_s(world, 6, 50, m)
    out.put((rank, m, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == res[1][2] == pytest.approx(2 * 6 * 50 / 0.015)


def test_reduce_max_without_process_group_is_identity():
    import bench
    assert bench.reduce_max(3.25, "cpu") == 3.25
    assert bench.tokens_per_s(1, 6, 10, 1.0) == pytest.approx(60000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        config = "tiny"
        steps = 1
        warmup = 0
    bench.reference_arm(A())            # returns at once on rank 1, printing nothing
    assert capsys.readouterr().out == ""
