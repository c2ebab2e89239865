"""Host logic of the multi-rank benchmark, on CPU with gloo (world size 2).

The path shards into independent replicas (one workload per GPU, no data
exchange); the only cross-rank operations are the barrier and the max over
ranks of the timed duration, which these tests exercise."""
from __future__ import annotations

import json
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.aggregate_max(1.5 + rank)          # rank 1 is the slow one
    dist.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slowest": slowest}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"r{r}.json"))["slowest"] for r in range(world)]
    assert got == [2.5, 2.5]


def test_job_value_is_weak_scaling_aggregate():
    f = bench.attention_flops(12, 4096)
    assert f == 4 * 12 * 4096 * 4096 * 64
    one = bench.job_value(f, 10, 1, 1e-3)
    two = bench.job_value(f, 10, 2, 1e-3)
    assert two == pytest.approx(2 * one)
    assert bench.job_value(f, 10, 2, 2e-3) == pytest.approx(one)


def test_reference_arm_prints_one_line(capsys, monkeypatch):
    monkeypatch.setenv("DERA_REF_BUDGET_S", "2")
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", "grid16"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", "grid16"]) == 0
    assert capsys.readouterr().out.strip() == ""
