"""Host logic of bench.py's multi-process mode, on CPU.

The decode step shards by stream with no collective, so N GPUs run N
independent replicas; the only cross-rank steps are the timing combination
(max over ranks) and the reference arm's rank-0-only rule.  The gather runs
here over a world-size-2 gloo group.
"""
from __future__ import annotations

import json
import os
import socket
import sys
import tempfile
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402


def test_combine_rank_times():
    ms, value = bench.combine_rank_times([2.0, 4.0], 64)
    assert ms == 4.0
    assert value == pytest.approx(2 * 64 / 4e-3)
    ms1, value1 = bench.combine_rank_times([0.5], 64)
    assert ms1 == 0.5 and value1 == pytest.approx(64 / 5e-4)


def test_dist_env(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "4")
    assert bench.dist_env() == (3, 4, 3)
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (3, 4, 1)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench as b
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        per_rank = b.max_over_ranks(1.5 + rank, world)  # each rank's mean step time (ms)
        ms, value = b.combine_rank_times(per_rank, 64)
        Path(out_dir, f"rank{rank}.json").write_text(json.dumps({"all": per_rank, "ms": ms, "value": value}))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(2, port, d), nprocs=2, join=True, start_method="spawn")
        res = [json.loads(Path(d, f"rank{r}.json").read_text()) for r in range(2)]
    for r in res:  # every rank sees both ranks' times and the same whole-job value
        assert r["all"] == [1.5, 2.5]
        assert r["ms"] == 2.5
        assert r["value"] == pytest.approx(2 * 64 / 2.5e-3)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
