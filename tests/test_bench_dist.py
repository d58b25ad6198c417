"""The multi-replica path of bench.py on CPU: two gloo ranks (no GPU).

The indexer has no exchange step, so N GPUs run N independent replicas; the
only cross-rank logic is the maximum of the per-rank timings (the slowest
replica sets the job's time), rank 0 alone printing the JSON line, and the
reference arm running on rank 0 only.
"""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], world, "cpu")
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.emit_line({"rank": rank, "value": got[0]}, rank)
        # the reference arm: ranks other than 0 exit 0 without work or output
        ref_out = io.StringIO()
        rc = None
        if rank != 0:
            with contextlib.redirect_stdout(ref_out):
                rc = bench.run_reference(type("A", (), {"gpus": world, "steps": 1, "warmup": 0})())
        q.put((rank, (w, r, lr), got, buf.getvalue(), rc, ref_out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_report():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, env, got, out, rc, ref_out = q.get(timeout=120)
        res[rank] = (env, got, out, rc, ref_out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        env, got, out, rc, ref_out = res[rank]
        assert env == (world, rank, rank)
        assert got == [2.0, 10.0, 3.5]  # element-wise maximum over the ranks
    assert res[0][2].strip().startswith("{") and '"rank": 0' in res[0][2]
    assert res[1][2] == ""  # only rank 0 prints
    assert res[1][3] == 0 and res[1][4] == ""


def test_single_rank_reduction_is_identity():
    import bench

    assert bench.max_over_ranks([1, 2.5], 1, "cpu") == [1.0, 2.5]
