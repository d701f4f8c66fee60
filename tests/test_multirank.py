"""Multi-process path of bench.py on CPU (gloo, world size 2).

Every row of the path is independent per KV head and per layer, so N GPUs run
N replicas (one layer each) with no collective on the data path; the only
collectives are the barrier around the timed region and the max over ranks of
the step time (the slowest rank sets the whole job's time).
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank)
    bench._barrier(ws)
    # each rank times a different step; the job's time is the slowest rank's
    t = bench._max_over_ranks(10.0 + 5.0 * rank, ws)
    out[rank] = t
    bench._barrier(ws)
    dist.destroy_process_group()


def test_two_ranks_max_step_time():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork of a multi-threaded test process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def _ref_worker(rank, world, port, out):
    # the reference arm prints only on rank 0; the other ranks exit without work
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import argparse
    import contextlib
    import io

    import bench
    buf = io.StringIO()
    if rank == 1:
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(argparse.Namespace(steps=1, warmup=0))
        out[rank] = (rc, buf.getvalue())


def test_reference_arm_other_ranks_exit_quietly():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork of a multi-threaded test process
    out = mgr.dict()
    mp.spawn(_ref_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[1] == (0, "")
