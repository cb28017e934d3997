"""Several replicas (bench.py --gpus N, one process per GPU, "replicas only":
the layer has no exchange step): the whole-job rate every rank computes, and
the reference arm's rank handling.  Run as world-size-2 gloo ranks on the CPU."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, ms: list, units: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        rate, ms_max = bench.job_rate(ms[rank], units, world, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"rate": rate, "ms": ms_max}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world, units, ms = 2, 300, [40.0, 50.0]
    mp.spawn(_rank_main, args=(world, _free_port(), ms, units, str(tmp_path)), nprocs=world,
             join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    # every rank sees the slowest rank's time, and the rate counts all ranks' units
    for g in got:
        assert g["ms"] == max(ms)
        assert g["rate"] == pytest.approx(world * units / (max(ms) * 1e-3), rel=1e-12)


def test_job_rate_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    rate, ms = bench.job_rate(25.0, 100, 1, "cpu")
    assert ms == 25.0 and rate == pytest.approx(4000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    """Under torchrun only rank 0 times the oracle; the others return at once."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 3, 3, 2

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
