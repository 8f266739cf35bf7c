"""The N>1 path of bench.py on CPU: world_size-2 gloo ranks (spawned processes) check that the job
time is the slowest rank's, that whole-job throughput counts every rank's work (weak scaling, no
data-path collective), and that only rank 0 runs the reference arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = [3.0, 5.0][rank]                           # this rank's device time (ms)
    mx = bench.max_over_ranks(t, world)
    val = bench.whole_job_tflops(1e12, 10, world, mx)
    q.put((rank, mx, val, bench._dist()))
    dist.barrier()
    dist.destroy_process_group()


def test_gloo_two_ranks_max_time_and_weak_scaling():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val, d in res:
        assert mx == 5.0                                # the slowest rank's time
        assert abs(val - 2 * 1e12 * 10 / 5e-3 / 1e12) < 1e-9
        assert d == (2, rank, rank)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1))

    class A:
        steps, warmup, gpus = 3, 3, 2
    assert bench.run_reference(A()) == 0
    assert called == [] and capsys.readouterr().out == ""
