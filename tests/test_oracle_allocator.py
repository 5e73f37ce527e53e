"""Pins for the reference allocator model.

"P3: native paged-KV continuous-batching sampler": Design / paged.py (LIFO free list,
refcounts, double-free guard, all-or-nothing ensure_capacity, shared blocks read-only for
everyone, owner included) and Evidence item 4 (10,000 randomized events with the books
checked after every event against refcounts recomputed from the live tables; more than 100
OOM events and more than 100 shared admits; pool fully free at the end).
"""
import numpy as np
import pytest

from oracle import allocator as al


def test_lifo_order_and_first_block():
    a = al.BlockAllocator(5)
    assert [a.alloc() for _ in range(3)] == [0, 1, 2]
    a.free(1)
    assert a.alloc() == 1          # most recently freed comes back first
    a.free(2)
    a.free(0)
    assert a.alloc() == 0
    assert a.alloc() == 2


def test_double_free_raises():
    a = al.BlockAllocator(2)
    b = a.alloc()
    a.free(b)
    with pytest.raises(al.DoubleFree):
        a.free(b)
    a.check_consistent()


def test_exhaustion_is_typed_and_changes_nothing():
    m = al.PagedCacheModel(4, 4)
    m.admit(0, 9)                                  # 3 blocks
    with pytest.raises(al.PoolExhausted):
        m.ensure_capacity(0, 17)                   # needs 2 more, 1 free
    assert len(m.tables[0]) == 3 and m.alloc.num_free == 1
    with pytest.raises(al.PoolExhausted):
        m.admit(1, 5)                              # needs 2
    assert 1 not in m.tables and m.alloc.num_free == 1
    m.check_consistent()


def test_shared_blocks_are_read_only_for_owner_too():
    m = al.PagedCacheModel(16, 4)
    m.admit(0, 10)                                 # blocks 0, 1, 2; 2 full blocks
    m.admit(1, 10, share_src=0, n_shared=2)
    assert m.tables[1][:2] == m.tables[0][:2]
    with pytest.raises(al.ReadOnlyBlock):
        m.slots(0, 4, 1)                           # owner writing into a shared block
    with pytest.raises(al.ReadOnlyBlock):
        m.slots(1, 0, 1)
    assert m.slots(0, 9, 1) == [m.tables[0][2] * 4 + 1]
    m.free_seq(0)
    assert m.slots(1, 4, 1)                        # refcount back to 1: writable
    m.free_seq(1)
    assert m.alloc.num_free == 16
    m.check_consistent()


def test_pool_guard_example_fits_exactly():
    """Prompt 3 + 6 new tokens at block size 4 caches 8 tokens: a 2-block pool suffices."""
    m = al.PagedCacheModel(2, 4)
    m.admit(0, 3 + 6 - 1)
    assert len(m.tables[0]) == 2 and m.alloc.num_free == 0


def property_run(model_cls_alloc=None, events=10_000, seed=0, num_blocks=48, bs=4):
    rng = np.random.default_rng(seed)
    m = al.PagedCacheModel(num_blocks, bs)
    live = {}
    next_id = 0
    stats = {"oom": 0, "shared": 0}
    for _ in range(events):
        op = rng.integers(0, 3) if live else 0
        if op == 0:                                  # admit, maybe sharing a prefix
            n = int(rng.integers(1, 40))
            src = None
            k = 0
            if live and rng.random() < 0.4:
                src = int(rng.choice(list(live)))
                full = live[src] // bs
                k = int(min(full, n // bs, rng.integers(0, 6)))
            try:
                m.admit(next_id, n, share_src=src if k else None, n_shared=k)
                live[next_id] = n
                stats["shared"] += k > 0
                next_id += 1
            except al.PoolExhausted:
                stats["oom"] += 1
        elif op == 1:                                # grow
            s = int(rng.choice(list(live)))
            n = live[s] + int(rng.integers(1, 20))
            try:
                m.ensure_capacity(s, n)
                live[s] = n
            except al.PoolExhausted:
                stats["oom"] += 1
        else:                                        # finish
            s = int(rng.choice(list(live)))
            m.free_seq(s)
            del live[s]
        m.check_consistent()
    for s in list(live):
        m.free_seq(s)
    m.check_consistent()
    assert m.alloc.num_free == num_blocks
    return stats


def test_property_run_10000_events():
    stats = property_run()
    assert stats["oom"] > 100 and stats["shared"] > 100


# --- mutants planted in the reference allocator: the books must catch each -------------

def _free_leaks(self, b):
    if self.ref[b] == 0:
        raise al.DoubleFree()
    self.ref[b] -= 1                      # never returns the block to the free list


def _free_double_appends(self, b):
    if self.ref[b] == 0:
        raise al.DoubleFree()
    self.ref[b] -= 1
    if self.ref[b] == 0:
        self.free_list.append(b)
        self.free_list.append(b)


def _no_incref(self, b):
    pass


def _no_double_free_guard(self, b):
    if self.ref[b] > 0:
        self.ref[b] -= 1
    if self.ref[b] == 0:
        self.free_list.append(b)


@pytest.mark.parametrize("attr,impl", [("free", _free_leaks), ("free", _free_double_appends),
                                       ("incref", _no_incref),
                                       ("free", _no_double_free_guard)])
def test_allocator_mutants_are_killed(monkeypatch, attr, impl):
    property_run(events=300, seed=3)        # control
    monkeypatch.setattr(al.BlockAllocator, attr, impl)
    caught = False
    try:
        property_run(events=300, seed=3)
        # the guard mutant survives a clean run; exercise the double free directly
        a = al.BlockAllocator(2)
        b = a.alloc()
        a.free(b)
        a.free(b)
        a.check_consistent()
    except (al.DoubleFree, al.Inconsistent, AssertionError):
        caught = True
    assert caught, "mutant survived"
