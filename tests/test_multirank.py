"""Multi-rank host logic on CPU with gloo (world sizes 2 and 3).

One call's (batch, head) problems are independent, so they are split into
contiguous ranges, one per rank, with no exchange while computing; a consumer
that needs the whole output gathers the slices afterwards.  These tests check
the partition (every problem exactly once, uneven counts), that the gathered
result equals a single-rank computation of the whole call, and the benchmark's
cross-rank steps (barrier, max over ranks of the timed duration)."""
from __future__ import annotations

import json
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from relative_position_bias_gb300 import shard


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


# --------------------------------------------------------------------------- BH partition of one call
@pytest.mark.parametrize("world", [1, 2, 3, 4, 5, 8])
def test_bh_ranges_tile_the_call(world):
    for BH in list(range(0, 40)) + [96, 192, 1001]:
        seen = []
        sizes = []
        for r in range(world):
            lo, hi = shard.bh_range(BH, r, world)
            assert 0 <= lo <= hi <= BH
            seen.extend(range(lo, hi))
            sizes.append(hi - lo)
        assert seen == list(range(BH))            # every (batch, head) exactly once, in order
        assert max(sizes) - min(sizes) <= 1


def test_bh_range_rejects_bad_ranks():
    with pytest.raises(ValueError):
        shard.bh_range(8, 2, 2)
    with pytest.raises(ValueError):
        shard.bh_range(8, 0, 0)
    with pytest.raises(ValueError):
        shard.bh_range(-1, 0, 1)


def _oracle_compute(q, k, v, th, tw, H, W, scale, **_):
    """CPU stand-in for one rank's device computation (the float64 oracle on the slice)."""
    out = oracle.fused(q.double().numpy(), k.double().numpy(), v.double().numpy(), th.double().numpy(),
                       tw.double().numpy(), H, W, scale)
    return torch.from_numpy(out)


def _shard_case(BH, H=3, W=4, d=8, seed=5):
    g = torch.Generator().manual_seed(seed)
    N = H * W
    q, k, v = (torch.randn(BH, N, d, generator=g) for _ in range(3))
    th, tw = 0.5 * torch.randn(2 * H - 1, d, generator=g), 0.5 * torch.randn(2 * W - 1, d, generator=g)
    return q, k, v, th, tw, H, W, d ** -0.5


def _shard_worker(rank: int, world: int, port: int, out_dir: str, BH: int):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, th, tw, H, W, scale = _shard_case(BH)
    part = shard.fused_shard(q, k, v, th, tw, H, W, scale, compute=_oracle_compute)
    full = shard.fused_shard(q, k, v, th, tw, H, W, scale, gather=True, compute=_oracle_compute)
    lo, hi = shard.bh_range(BH, rank, world)
    torch.save({"lo": lo, "hi": hi, "part": part, "full": full}, os.path.join(out_dir, f"s{rank}.pt"))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,BH", [(2, 7), (3, 7), (3, 2), (2, 12)])
def test_sharded_call_gathers_to_the_single_rank_result(tmp_path, world, BH):
    mp.spawn(_shard_worker, args=(world, _free_port(), str(tmp_path), BH), nprocs=world, join=True)
    q, k, v, th, tw, H, W, scale = _shard_case(BH)
    want = _oracle_compute(q, k, v, th, tw, H, W, scale)
    got = [torch.load(tmp_path / f"s{r}.pt") for r in range(world)]
    covered = []
    for r, rec in enumerate(got):
        assert torch.equal(rec["full"], want), f"rank {r}: gathered output differs from the single-rank call"
        assert torch.equal(rec["part"], want[rec["lo"]:rec["hi"]])
        covered.extend(range(rec["lo"], rec["hi"]))
    assert covered == list(range(BH))


# --------------------------------------------------------------------------- the backward's exchange step
def _oracle_backward(q, k, v, th, tw, out, lse, dout, H, W, scale, **_):
    """CPU stand-in for one rank's backward (the float64 oracle on the slice; out and lse unused)."""
    g = oracle.fused_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(), th.double().numpy(),
                              tw.double().numpy(), H, W, scale, dout.double().numpy())
    return tuple(torch.from_numpy(x) for x in g)


def _bwd_worker(rank: int, world: int, port: int, out_dir: str, BH: int):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, th, tw, H, W, scale = _shard_case(BH)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(11))
    out = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2])
    g = shard.fused_backward_shard(q, k, v, th, tw, out, lse, dout, H, W, scale, compute=_oracle_backward)
    lo, hi = shard.bh_range(BH, rank, world)
    torch.save({"lo": lo, "hi": hi, "g": g}, os.path.join(out_dir, f"b{rank}.pt"))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,BH", [(2, 7), (3, 5), (3, 2)])
def test_sharded_backward_sums_the_table_gradients(tmp_path, world, BH):
    """dq, dk, dv of a rank are its slice of the whole call's; the table gradients, summed over the
    ranks' partials in rank order, equal the whole call's and are the same on every rank."""
    mp.spawn(_bwd_worker, args=(world, _free_port(), str(tmp_path), BH), nprocs=world, join=True)
    q, k, v, th, tw, H, W, scale = _shard_case(BH)
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(11))
    want = _oracle_backward(q, k, v, th, tw, None, None, dout, H, W, scale)
    recs = [torch.load(tmp_path / f"b{r}.pt") for r in range(world)]
    for r, rec in enumerate(recs):
        lo, hi = rec["lo"], rec["hi"]
        for i in range(3):
            assert torch.equal(rec["g"][i], want[i][lo:hi]), f"rank {r}: gradient {i} is not its slice"
        for i in (3, 4):
            assert torch.allclose(rec["g"][i], want[i], rtol=0, atol=1e-12)
            assert torch.equal(rec["g"][i], recs[0]["g"][i])   # every rank holds the same sum
