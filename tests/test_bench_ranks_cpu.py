"""bench.py's bookkeeping on CPU.  Multi-replica: with two gloo ranks, every rank gets the
element-wise maximum of the ranks' times (the slowest replica defines the job) and the
whole-job rate counts every rank's units over that time; the replicas share nothing else
(the decoder path itself has no collective).  Roofline: the profiled DRAM traffic is
reported only for the kernel sources it was captured with."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [1.0 + rank, 5.0 - 2 * rank, 0.25 * (rank + 1)]
        got = bench.reduce_max_over_ranks(times, world, "cpu")
        out[rank] = (got, bench.whole_job_rate(world, 64 * 3, got[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_and_count_every_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(world):
            got, rate = out[r]
            assert got == [2.0, 5.0, 0.5]
            assert rate == pytest.approx(world * 64 * 3 / 2.0)


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks([3, 1.5], 1, "cpu") == [3.0, 1.5]
    assert bench.whole_job_rate(1, 100, 4.0) == 25.0


def test_profiled_traffic_only_while_the_kernel_sources_match(tmp_path, monkeypatch):
    """The decode roofline's DRAM traffic comes from an ncu capture: bench.py reports it only
    while the decode kernel's source files hash to the value recorded with that capture, and
    null once they change (or for a workload never captured)."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel source at the capture\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "DECODE_KERNEL_SOURCES", ("kernel.cu",))
    monkeypatch.setattr(bench, "PROFILED_DECODE_TRAFFIC", {"w": (bench.decode_sources_sha(), 1234)})
    assert bench.profiled_decode_traffic("w") == 1234
    assert bench.profiled_decode_traffic("other") is None
    src.write_text("// kernel source changed since the capture\n")
    assert bench.profiled_decode_traffic("w") is None
