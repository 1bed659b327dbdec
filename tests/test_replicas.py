"""Replicas: `bench.py --gpus N` runs N independent batches, one per rank, and
reduces only the timing (the slowest rank's time; bytes of all ranks). No data
crosses ranks. The host logic runs here with two gloo ranks on the CPU."""
import contextlib
import io
import json
import os
import socket
import types

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workload as W
        # the job's time is the slowest rank's
        t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        # each rank draws its own batch
        cfg = W.CONFIGS["llama3_8b_b32"]
        wl = W.make_workload(cfg, seed=bench.replica_seed(cfg.seed, rank))
        # the reference arm: rank 0 alone prints its line, the others exit at once
        args = types.SimpleNamespace(config="tiny_1layer", steps=1, warmup=0, window=0)
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args)
        dist.barrier()
        q.put((rank, t, wl.context_lens.tolist(), buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_time_only_and_draw_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=300) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    (r0, t0, ctx0, out0), (r1, t1, ctx1, out1) = res
    assert t0 == t1 == 15.0
    assert ctx0 != ctx1  # independent batches
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert out1 == ""


def test_whole_job_value_counts_every_rank():
    import bench
    assert bench.whole_job_gbs(1, 10 ** 9, 1.0) == pytest.approx(1000.0)
    assert bench.whole_job_gbs(4, 10 ** 9, 2.0) == pytest.approx(2000.0)
    assert bench.replica_seed(1002, 0) == 1002 and bench.replica_seed(1002, 3) == 4002
