"""Replica path of bench.py on CPU (not gpu): two gloo ranks, each with its own
elapsed time, agree on the slowest one, and the whole-job value counts the
units of both replicas over that time.  The quantized linear has no exchange
step, so replicas are the multi-GPU form; this covers their host logic."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed = [0.75, 1.25][rank]
    m = bench.max_over_ranks(elapsed)
    v = bench.whole_job_value(units_per_step=1e9, steps=10, world=world, elapsed_max=m, unit_scale=1e9)
    dist.barrier()
    out[rank] = (m, v)
    dist.destroy_process_group()


def test_two_replicas_agree_on_slowest_and_sum_units():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    m, v = res[0]
    assert m == 1.25
    assert v == pytest.approx(1e9 * 10 * 2 / 1.25 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.whole_job_value(2e9, 4, 1, 2.0, 1e9) == pytest.approx(4.0)
