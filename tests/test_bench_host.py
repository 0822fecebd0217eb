"""Host logic of bench.py on CPU: the whole-job aggregation over ranks (gloo,
world size 2) and the single-process path."""

from __future__ import annotations

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, rows, secs, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        value, sec, total = bench.aggregate(rows[rank], secs[rank])
        out[rank] = torch.tensor([value, sec, total], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


def test_aggregate_single_process():
    value, sec, total = bench.aggregate(64.0, 0.5)
    assert (value, sec, total) == (128.0, 0.5, 64.0)


@pytest.mark.timeout(120)
def test_aggregate_over_two_gloo_ranks():
    """value = rows of all ranks / the slowest rank's time, on every rank."""
    world = 2
    rows = [32.0, 32.0]
    secs = [0.25, 0.40]
    out = torch.zeros(world, 3, dtype=torch.float64).share_memory_()
    mp.spawn(_rank_main, args=(world, _free_port(), rows, secs, out), nprocs=world, join=True)
    for r in range(world):
        value, sec, total = out[r].tolist()
        assert total == 64.0
        assert sec == 0.40
        assert value == pytest.approx(64.0 / 0.40)


def test_kernel_mode_is_parsed(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--kernel", "topk", "--steps", "2", "--warmup", "1"])
    a = bench.parse()
    assert a.kernel == "topk" and a.steps == 2 and a.warmup == 1 and a.gpus == 1


def test_default_workload_is_the_largest_configuration(monkeypatch):
    """With no flags the contract line times the ragged fp8 sweep at B = 256;
    --config selects another configuration."""
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    s = bench.workload_spec(a)
    assert (s.B, s.dtype, s.length_law, s.L_lo, s.L_hi, s.topk, s.H) == (
        256, "fp8_e4m3", "loguniform", 4096, 131072, 2048, 32)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "1"])
    s1 = bench.workload_spec(bench.parse())
    assert (s1.B, s1.L, s1.dtype) == (32, 32768, "bf16")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "4", "--batch", "64"])
    assert bench.workload_spec(bench.parse()).B == 64


def test_algorithmic_bytes_closed_form():
    """Per-kernel algorithmic bytes of a tiny bf16 workload, written out."""
    from workloads import config_spec, make_workload

    wl = make_workload(config_spec(1, B=2, L=300, H=16))
    b = bench.algorithmic_bytes(wl)
    L, k, H = 300, 2048, 16
    assert b["indexer"] == 2 * (L * 256 + 5 * 4) + 2 * (64 * 128 * 2 + 64 * 4)
    assert b["topk"] == 2 * (L * 4 + k * 4 + 4)
    assert b["mla"] == 2 * (L * 1152 + k * 4 + H * 576 * 2 + H * 512 * 4 + H * 4)


def test_single_thread_oracle_figure_on_config0():
    """The CPU baseline also reports the oracle on configuration 0 with one
    BLAS thread (run in a child process, so that the thread count holds)."""
    import bench

    d = bench.single_thread_config0(0.3)
    assert "error" not in d, d
    assert d["cores"] == 1 and d["value"] > 0 and d["unit"] == bench.UNIT
