"""The N > 1 benchmark path on CPU: two gloo ranks run independent replicas
and meet only for a barrier and a max-reduce of their timings (no data-path
collective).  Checks that every rank sees the slowest rank's time and that
the whole-job throughput counts both replicas' work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_setup()
        bench.barrier(w)
        slowest = bench.max_over_ranks(10.0 + rank, w, "cpu")  # rank 1 is slower
        gbs = bench.replica_throughput(16_814_080, slowest, w)
        bench.barrier(w)
        q.put((r, lr, w, slowest, gbs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_count_all_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [g[0] for g in got] == [0, 1] and all(g[2] == 2 for g in got)
    for _, _, _, slowest, gbs in got:
        assert slowest == 11.0
        assert gbs == pytest.approx(2 * 16_814_080 / 11e-6 / 1e9)


def test_reference_arm_only_runs_on_rank_zero(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 0
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
