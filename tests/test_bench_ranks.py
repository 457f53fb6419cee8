"""Multi-rank helpers of bench.py on CPU: two gloo ranks (no GPU).

The forward path has no collective (units are independent, so N GPUs run N replicas);
the only cross-rank steps are the barrier around the timed region and the maximum of
the per-rank step time.  This checks both, and that the reference arm prints nothing
on ranks other than 0.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)          # per-rank step times 1.5 and 2.5 ms
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 2.5


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_is_silent_off_rank_zero(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload, steps, warmup, oracle_threads = "tiny", 1, 3, 0
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


def test_both_arms_share_metric_and_config():
    sys.path.insert(0, ROOT)
    import bench
    from gated_delta_rule_36_gb300.inputs import workload
    w = workload("packed64")
    cfg = bench.bench_config(w, 1)
    assert cfg["workload"] == "packed64" and cfg["tokens"] == w.total_tokens and cfg["heads"] == 64
    assert "GB300" in bench.METRIC


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """The reference arm (the oracle on host cores) prints one JSON line with the keys the
    benchmark contract names, its e2e and cpu_baseline objects describing the same run."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")

    class Args:
        workload, steps, warmup, oracle_threads = "tiny", 1, 3, 0
    bench.run_reference(Args())
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"] == bench.bench_config(bench_workload("tiny"), 1)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def bench_workload(name):
    from gated_delta_rule_36_gb300.inputs import workload
    return workload(name)
