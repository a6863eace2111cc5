"""The replica path of bench.py across two CPU ranks (gloo): every rank receives the
slowest rank's time, and the job's throughput counts every rank's units over it."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info()[:2] == (rank, world)
        ms_local = [3.0, 5.0, 4.0][rank]
        ms = bench.max_over_ranks(ms_local, world, device="cpu")
        value = bench.job_throughput(16 * 100, world, ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms} {value}")
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_job_throughput(tmp_path, world):
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        ms, value = map(float, (tmp_path / f"rank{r}.txt").read_text().split())
        assert ms == 5.0                                   # the slowest replica
        assert value == pytest.approx(world * 16 * 100 / 5e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.job_throughput(10, 1, 1000.0) == pytest.approx(10.0)
