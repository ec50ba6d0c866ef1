"""The multi-replica host logic of bench.py on CPU, with two gloo ranks (no GPU): the job's time is the
slowest rank's, its throughput sums every replica's tokens, and the reference arm prints on rank 0 only.
The method has no data-path collective: each rank runs a whole replica; these are the only exchanges."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        slowest = bench.max_over_ranks(1.0 + 0.5 * rank, "cpu")  # per-rank step times 1.0, 1.5 ms
        dist.barrier()
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0, "ref_heads": 1})()) if rank else "skip"
        out[rank] = (slowest, bench.job_tokens_per_s(slowest, world), ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_replicas():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    import bench
    for rank in range(world):
        slowest, value, ref = res[rank]
        assert slowest == pytest.approx(1.5)  # both ranks see the slowest rank's time
        assert value == pytest.approx(world * 2 * bench.B * bench.N / 1.5e-3)
    assert res[1][2] is None  # the reference arm prints nothing on rank 1


def test_without_a_process_group_the_local_time_stands():
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.job_tokens_per_s(1.0, 1) == pytest.approx(2 * bench.B * bench.N / 1e-3)
