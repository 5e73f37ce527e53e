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


def _replica_worker(rank, world, port, out):
    """One replica: its own sequence set, its own allocator over its own pool, its own step
    metadata and plan, all through the C ABI (host calls only), checked against the oracle's
    allocator model and slot mapping. The ranks exchange nothing but the final summaries."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from continuous_batching_gb300 import binding as bd
    from oracle import allocator as al
    import oracle.paged_attention as pa
    rng = np.random.default_rng(100 + rank)
    bs, nb, B = 16, 512, 12
    shape = bd.Shape.make(32, 8, 128, bs, nb)
    alloc = bd.Allocator(nb, bs)
    model = al.PagedCacheModel(nb, bs)
    prompt = rng.integers(20, 400, size=B)
    for s in range(B):
        alloc.admit(s, int(prompt[s]))
        model.admit(s, int(prompt[s]))
    # one mixed step: sequences 0..3 prefill a chunk, the others decode one token
    n_new = np.where(np.arange(B) < 4, np.minimum(prompt, 64), 1).astype(np.int32)
    ctx = np.where(np.arange(B) < 4, n_new, prompt + 1).astype(np.int32)
    for s in range(4, B):
        alloc.ensure_capacity(s, int(ctx[s]))
        model.ensure_capacity(s, int(ctx[s]))
    max_blocks = int((ctx.max() + bs - 1) // bs)
    cu, slots, table = alloc.build_step(np.arange(B), ctx, n_new, max_blocks)
    alloc.check_consistent()
    want_table = np.full((B, max_blocks), -1, np.int32)
    for s in range(B):                         # the entries that cover ctx, -1 after
        t = model.tables[s][:(int(ctx[s]) + bs - 1) // bs]
        want_table[s, :len(t)] = t
    ok_table = np.array_equal(table, want_table)
    ok_slots = np.array_equal(slots, pa.slot_mapping(table, cu, ctx, bs)) and np.array_equal(
        slots, np.concatenate([model.slots(s, int(ctx[s] - n_new[s]), int(n_new[s]))
                               for s in range(B)]))
    items = bd.pa_plan_step(shape, cu, ctx)
    # every (row, KV head, split) exactly once
    seen = set()
    for it in items:
        for t in range(it["q_start"], it["q_start"] + it["n_q"]):
            for sp in range(it["split"], it["split"] + max(int(it["n_splits"]), 1)):
                key = (t, int(it["kv_head"]), sp)
                assert key not in seen
                seen.add(key)
    rows = np.searchsorted(cu, np.arange(int(cu[-1])), side="right") - 1
    need = {(t, h, sp) for t in range(int(cu[-1])) for h in range(8)
            for sp in range((int(ctx[rows[t]]) - int(cu[rows[t] + 1]) + t) // bd.PA_SPLIT_TOKENS + 1)}
    summary = (ok_table, ok_slots, seen == need, int(cu[-1]), int(ctx.sum()), alloc.num_free,
               model.alloc.num_free)
    got = [None] * world
    dist.all_gather_object(got, summary)
    out[rank] = got
    dist.destroy_process_group()


def test_two_gloo_replicas_plan_their_own_steps_through_the_c_abi():
    from continuous_batching_gb300 import build
    build.build()
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_replica_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]                      # both ranks saw both summaries
    for ok_table, ok_slots, ok_plan, T, kv, free_lib, free_model in out[0]:
        assert ok_table and ok_slots and ok_plan
        assert free_lib == free_model
    assert out[0][0][4] != out[0][1][4]          # different sequence sets


def test_single_process_is_identity():
    import bench
    assert bench.combine_ranks(3.0, 7.0) == (3.0, 7.0)
