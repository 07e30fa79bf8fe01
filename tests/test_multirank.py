"""The multi-GPU launch of bench.py is replicas only: each rank runs its own
batch, a barrier brackets the timed region, the slowest rank's time sets the
job time and the job throughput counts every rank's tokens.  These host-side
pieces run here as two gloo ranks on the CPU (no GPU, no NCCL)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_replicas("gloo")
    dist.barrier()
    ms = bench.max_over_ranks(dist, 1.5 + rank, "cpu")  # rank r took 1.5 + r ms per step
    value = bench.job_throughput(world, 4096, ms)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms} {value}")
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank_and_count_every_rank(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        ms, value = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        assert ms == pytest.approx(2.5)                     # max over ranks
        assert value == pytest.approx(world * 4096 / 2.5e-3)  # all ranks' tokens / slowest time


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_replicas("gloo") is None
    assert bench.max_over_ranks(None, 3.25, "cpu") == 3.25
    assert bench.job_throughput(1, 1000, 2.0) == pytest.approx(5e5)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # under torchrun every rank but 0 exits at once without work or output
    monkeypatch.setenv("RANK", "1")
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        config, T, steps, warmup, ref_sample = "mixtral", 4096, 1, 3, 16

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""
