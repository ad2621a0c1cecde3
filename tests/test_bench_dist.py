"""bench.py's multi-rank logic on the CPU with gloo, world size 2: every rank runs
its own layer (weak scaling, no data-path collective), the time is the max over
ranks, the whole-job value counts every rank's work, and the reference arm runs
on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from mixed_precision_attention_gb300 import synth
    w = synth.WORKLOADS[bench.WORKLOAD]
    got = dict(setup=bench.dist_setup(),
               ms=bench.max_over_ranks(1.0 + 2.0 * rank, world, torch.device("cpu")),
               seed=bench.rank_layer_seed(w, rank))
    bench.barrier(world)
    out.put((rank, got))
    dist.destroy_process_group()


def test_two_ranks_with_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0]["setup"] == (2, 0, 0) and res[1]["setup"] == (2, 1, 1)
    assert res[0]["ms"] == res[1]["ms"] == 3.0          # the slowest rank's time, on every rank
    assert res[0]["seed"] != res[1]["seed"]             # each rank its own layer


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1, 3.0e12, 2.0)
    assert one == pytest.approx(1500.0)
    assert bench.whole_job_tflops(4, 3.0e12, 2.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        gpus, steps, warmup = 2, 1, 0
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
