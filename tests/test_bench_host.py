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


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference times the oracle on the host and prints one
    JSON line with the reference arm's keys (tiny workload: a few seconds)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                       env={**os.environ, "RANK": "0"})
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["steps"] == 2 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"]


def test_committed_traffic_only_while_the_kernel_sources_match(monkeypatch, tmp_path):
    """roofline.traffic comes from the committed ncu record only while the
    hashed kernel sources are the ones it was captured on; otherwise null."""
    srcs = ["a.cu", "b.cuh"]
    for name in srcs:
        (tmp_path / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", srcs)
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        f"# workload bytes hash\nqwen_q4 123456 {h}\nqwen_q2 999 0000000000000000\n")
    assert bench.committed_traffic("qwen_q4") == 123456.0
    assert bench.committed_traffic("qwen_q2") is None          # captured on other sources
    assert bench.committed_traffic("stack48") is None          # no record
    (tmp_path / "b.cuh").write_text("// b.cuh, changed\n")
    assert bench.committed_traffic("qwen_q4") is None
