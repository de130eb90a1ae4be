"""The multi-GPU path is replicas only (requests and kv heads are
independent; no exchange step): N ranks each run the whole workload and the
benchmark reports the bytes of all ranks over the slowest rank's time. This
checks that host logic with two gloo ranks on the CPU: the max over ranks,
the whole-job figure, and that the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + 3.0 * rank  # rank 1 is the slow replica
        job_ms = bench.max_over_ranks(ms, torch.device("cpu"))
        results[rank] = (job_ms, bench.whole_job_gbs(1e9, world, job_ms))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0][0] == got[1][0] == 5.0          # every rank sees the slowest time
    assert got[0][1] == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_single_process_keeps_its_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.whole_job_gbs(2e9, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_rank_nonzero_does_no_work():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.argparse.Namespace(warmup=3, steps=1, reference_seconds=0.1)
    assert bench.run_reference(args, rank=1, world=2) is None

