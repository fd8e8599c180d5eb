"""Host logic of the N > 1 benchmark path on CPU: two `gloo` ranks (one process each, as under
torchrun). Every rank runs an independent replica (no collective on the data path); the job's
step time is the maximum over ranks and its throughput the sum of the replicas' work."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from attention_relative_position_gb300 import workloads as wl
        w = wl.WORKLOADS[1]
        step_ms = bench.max_over_ranks(1.0 + 2.5 * rank, "cpu")
        cfg = bench.workload_config(w, world, "test")
        value = bench.job_tflops(3.5 * w.fwd_flops(), world, step_ms)
        q.put((rank, step_ms, cfg["global_tokens"], cfg["parallelism"], value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_replica_config():
    from attention_relative_position_gb300 import workloads as wl
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = wl.WORKLOADS[1]
    slowest = 1.0 + 2.5  # rank 1's step time
    for rank, step_ms, tokens, par, value in res:
        assert step_ms == pytest.approx(slowest)
        assert tokens == 2 * w.total_tokens
        assert par == "replicas x2"
        assert value == pytest.approx(3.5 * w.fwd_flops() * 2 / slowest / 1e9)


def test_single_process_keeps_its_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, "cpu") == 4.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    # rank 1 of 2 returns at once (before reading its arguments) and prints nothing
    bench.run_reference(None, 1, 2)
    assert capsys.readouterr().out == ""
