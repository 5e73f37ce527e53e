"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own batch (the path
shards by sequence with no exchange), whole-job value = units of all ranks / slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from continuous_batching_gb300 import workloads as wl
    st = wl.make_config("decode", with_pool=False, seed=bench.rank_seed("decode", rank))
    units = float(bench.kv_bytes(st))
    t, u = bench.combine_ranks(10.0 + 5.0 * rank, units, dist, "cpu")
    out[rank] = (t, u, units, int(st.ctx_lens.sum()))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_sum_units():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    t0, u0, a, c0 = out[0]
    t1, u1, b, c1 = out[1]
    assert t0 == t1 == 15.0                       # slowest rank
    assert u0 == u1 == a + b                      # all ranks' units
    assert c0 != c1                               # each rank drew its own batch


def test_single_process_is_identity():
    import bench
    assert bench.combine_ranks(3.0, 7.0) == (3.0, 7.0)
