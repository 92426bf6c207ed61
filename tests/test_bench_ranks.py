"""Host side of the benchmark's multi-GPU path, on CPU with two gloo ranks.

The layer's data path does not exchange data between GPUs: N ranks run N
independent replicas, and the benchmark reports the tokens of all ranks over
the slowest rank's time.  These checks run that reduction (and the reference
arm's rank gating) in two processes on the host, with no GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], torch.device("cpu"))
        value = bench.replica_tokens_per_s(world, 4096, ms)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    times = [0.431, 0.447]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        ms, value = res[rank]
        assert ms == pytest.approx(max(times))                 # every rank sees the slowest
        assert value == pytest.approx(world * 4096 / (max(times) * 1e-3))


def test_max_over_ranks_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25
    assert bench.replica_tokens_per_s(1, 4096, 0.5) == pytest.approx(4096 / 0.5e-3)


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    """Under torchrun the reference arm (the CPU oracle) runs on rank 0 alone;
    the other ranks return at once without work."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 3, 3

    assert bench.run_reference(Args()) is None
