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
        workload, steps, warmup = "tiny", 1, 3
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
