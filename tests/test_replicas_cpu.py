"""The multi-rank host logic of a run on N GPUs (replicas: no exchange on the
data path), exercised with world_size-2 gloo ranks on the CPU: the barrier,
the maximum over ranks of the timed region, and the whole-job rate."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from quantized_speculative_decoding_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = replicas.world_rank_local()
    replicas.barrier(w)
    # each rank "measured" different times; every rank must see the maximum
    mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
    got = replicas.max_over_ranks(mine, w, "cpu")
    replicas.barrier(w)
    dist.destroy_process_group()
    q.put((r, l, w, got))


def test_two_gloo_ranks_agree_on_max_times():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _, _ in res) == [0, 1]
    for r, l, w, got in res:
        assert w == world and l == r
        assert got == [2.0, 5.0, 0.5]


def test_single_rank_is_a_no_op(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert replicas.world_rank_local() == (1, 0, 0)
    replicas.barrier(1)
    assert replicas.max_over_ranks([3, 1.5], 1, "cpu") == [3.0, 1.5]


def test_whole_job_rate_is_weak_scaling():
    # N ranks, each the same work: units of all ranks over the slowest rank's time
    assert replicas.whole_job_rate(1, 100.0, 2.0) == pytest.approx(50.0)
    assert replicas.whole_job_rate(4, 100.0, 2.0) == pytest.approx(200.0)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
