"""Host logic of bench.py for N > 1 replicas: max over ranks and the whole-job
value, run as two gloo ranks on the CPU (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms for the kernel steps and 30 - r ms end to end
        ms, e2e = bench.max_over_ranks([(rank + 1) * 10.0, 30.0 - rank], torch.device("cpu"), world)
        out[rank] = (ms, e2e, bench.job_gbs(1e9, 4, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, e2e, gbs = res[r]
        assert ms == 20.0 and e2e == 30.0          # the slowest rank decides
        assert gbs == pytest.approx(1e9 * 4 * 2 / 0.020 / 1e9)   # all ranks' bytes


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu"), 1) == [3.0, 4.0]
    assert bench.job_gbs(35389440 * 64, 100, 1, 139.3) == pytest.approx(1626.0, rel=1e-3)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    ns = type("A", (), {"workload": "tiny", "chain": 1, "steps": 1, "warmup": 0, "gpus": 2})()
    assert bench.run_reference(ns) == 0
