"""The C++ host allocator of libpagedattn against the oracle's reference allocator model,
event by event (bit-exact tables, refcounts and free counts), plus its typed errors and the
one-step metadata builder. CPU only."""
import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from oracle import allocator as al


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import os
    if not os.path.exists(bd.LIB_PATH):
        from continuous_batching_gb300 import build
        build.build()
    bd.load()


def test_lifo_order_matches_reference():
    a = bd.Allocator(6, 4)
    r = al.BlockAllocator(6)
    seq = []
    for op in ["a", "a", "a", "f1", "a", "f0", "f2", "a", "a"]:
        if op == "a":
            seq.append((a.alloc(), r.alloc()))
        else:
            b = int(op[1])
            a.free(b)
            r.free(b)
    assert all(x == y for x, y in seq)
    assert seq[0][0] == 0
    a.close()


def test_typed_errors():
    a = bd.Allocator(2, 4)
    b = a.alloc()
    a.free(b)
    with pytest.raises(bd.DoubleFree):
        a.free(b)
    a.admit(1, 8)
    with pytest.raises(bd.PoolExhausted):
        a.ensure_capacity(1, 9)
    assert a.table(1) == [0, 1] or len(a.table(1)) == 2
    with pytest.raises(bd.PoolExhausted):
        a.admit(2, 1)
    a.check_consistent()
    a.close()


def test_readonly_shared_blocks():
    a = bd.Allocator(16, 4)
    a.admit(0, 10)
    a.admit(1, 10, share_src=0, n_shared=2)
    assert a.table(1)[:2] == a.table(0)[:2]
    assert a.refcount(a.table(0)[0]) == 2
    with pytest.raises(bd.ReadOnlyBlock):
        a.slots(0, 4, 1)
    with pytest.raises(bd.ReadOnlyBlock):
        a.build_step([1], [10], [3], 4)          # positions 7..9: 7 is in the shared block 1
    cu, slots, table = a.build_step([1, 0], [10, 10], [2, 1], 4)
    assert cu.tolist() == [0, 2, 3]
    t1 = a.table(1)
    assert slots.tolist() == [t1[2] * 4 + 0, t1[2] * 4 + 1, a.table(0)[2] * 4 + 1]
    assert table[0, :3].tolist() == t1 and table[0, 3] == -1
    a.free_seq(0)
    a.free_seq(1)
    assert a.num_free == 16
    a.check_consistent()
    a.close()


def test_pool_guard_example():
    """Prompt 3 + 6 new at block 4: 8 cached tokens fit a 2-block pool exactly."""
    a = bd.Allocator(2, 4)
    a.admit(0, pa.cached_tokens(3, 6))
    assert len(a.table(0)) == pa.blocks_needed(8, 4) == 2 and a.num_free == 0
    a.close()


def test_property_run_against_reference_10000_events():
    rng = np.random.default_rng(7)
    nb, bs = 48, 4
    cpp = bd.Allocator(nb, bs)
    ref = al.PagedCacheModel(nb, bs)
    live = {}
    nid = 0
    oom = shared = 0
    for ev in range(10_000):
        op = rng.integers(0, 3) if live else 0
        if op == 0:
            n = int(rng.integers(1, 40))
            src, k = None, 0
            if live and rng.random() < 0.4:
                src = int(rng.choice(list(live)))
                k = int(min(live[src] // bs, n // bs, rng.integers(0, 6)))
            r_err = c_err = None
            try:
                ref.admit(nid, n, share_src=src if k else None, n_shared=k)
            except al.PoolExhausted:
                r_err = "oom"
            try:
                cpp.admit(nid, n, share_src=src if k else None, n_shared=k)
            except bd.PoolExhausted:
                c_err = "oom"
            assert r_err == c_err
            if r_err is None:
                live[nid] = n
                shared += k > 0
                nid += 1
            else:
                oom += 1
        elif op == 1:
            s = int(rng.choice(list(live)))
            n = live[s] + int(rng.integers(1, 20))
            r_err = c_err = None
            try:
                ref.ensure_capacity(s, n)
            except al.PoolExhausted:
                r_err = "oom"
            try:
                cpp.ensure_capacity(s, n)
            except bd.PoolExhausted:
                c_err = "oom"
            assert r_err == c_err
            if r_err is None:
                live[s] = n
            else:
                oom += 1
        else:
            s = int(rng.choice(list(live)))
            ref.free_seq(s)
            cpp.free_seq(s)
            del live[s]
        cpp.check_consistent()
        ref.check_consistent()
        assert cpp.num_free == ref.alloc.num_free
        if ev % 97 == 0:
            for s in live:
                assert cpp.table(s) == ref.tables[s]
            for b in range(nb):
                assert cpp.refcount(b) == ref.alloc.ref[b]
    for s in list(live):
        cpp.free_seq(s)
    cpp.check_consistent()
    assert cpp.num_free == nb
    assert oom > 100 and shared > 100
    cpp.close()
