"""The multi-GPU path of bench.py, on the CPU.

A batch-1 decode stream does not shard, so N GPUs run N independent
replicas: each rank times its own steps between barriers, and rank 0
reports the slowest rank's time and the tokens of all ranks.  These tests
run that host logic as two gloo ranks (world size 2, spawned processes,
rendezvous on 127.0.0.1), and check that the reference arm's other ranks
leave without work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier()
        # rank r: 10 + r ms for 100 * (r + 1) tokens
        ms, units = bench.reduce_over_ranks(10.0 + rank, 100.0 * (rank + 1))
        bench.barrier()
        out.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_time_and_all_tokens():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see max time 11 ms and 100 + 200 tokens
    assert got == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_reduce_is_identity_without_a_process_group():
    import bench
    assert bench.reduce_over_ranks(3.5, 7.0) == (3.5, 7.0)


def test_reference_arm_other_ranks_leave_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
