"""The N > 1 path of the bench on the CPU: replicas, one per rank, with no collective
on the data path.  Two gloo ranks check the cross-rank timing: every rank ends with
the slowest rank's time, and the whole-job throughput counts every rank's units
over that time.  The library's calls take no part: nothing of them crosses ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        ms = bench.max_over_ranks(dist, times[rank], device="cpu")
        rate = bench.job_rate(world, 231 * 32, ms)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{ms!r} {rate!r}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate(tmp_path):
    times = [9.25, 9.75]   # ms per step of each replica
    mp.start_processes(_rank_main, args=(2, _free_port(), times, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [tuple(float(x) for x in (tmp_path / f"r{r}.txt").read_text().split()) for r in range(2)]
    assert got[0] == got[1]
    ms, rate = got[0]
    assert ms == max(times)
    assert rate == pytest.approx(2 * 231 * 32 / (max(times) / 1e3))


def test_without_a_process_group_the_rank_keeps_its_own_time():
    import bench
    assert bench.max_over_ranks(None, 4.5) == 4.5
    assert bench.job_rate(1, 100, 1000.0) == pytest.approx(100.0)
