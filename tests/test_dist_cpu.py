"""The multi-GPU bookkeeping of bench.py on CPU: two gloo ranks (replicas).

bench.py runs one replica per GPU under torchrun; the job's time is the
slowest rank's and the throughput counts every rank's units. Here two CPU
processes stand in for two ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slow replica
        m = bench.max_over_ranks(ms)
        rate = bench.job_rate(16, m, world)
        dist.barrier()
        results[rank] = (m, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_rate():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(results)
    # every rank sees the slowest rank's time, and the rate counts both ranks
    assert got[0] == got[1] == (15.0, pytest.approx(16 * 2 * 1000.0 / 15.0))


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rate(1, 2.0, 1) == 500.0


def test_host_cpu_record(tmp_path):
    import bench
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nmodel name\t: Some CPU @ 2.0GHz\nflags\t: fpu\n")
    assert bench.host_cpu(str(x86))["model"] == "Some CPU @ 2.0GHz"
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\n"
                   "CPU part\t: 0xd4f\n\nprocessor\t: 1\nCPU implementer\t: 0x41\n")
    rec = bench.host_cpu(str(arm))
    assert rec["model"] == "implementer 0x41 part 0xd4f" and rec["nproc"] >= 1
    assert bench.host_cpu(str(tmp_path / "missing"))["model"]
