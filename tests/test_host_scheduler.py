"""The C++ scheduler and the allocator's trim / fork / copy-on-write, event by event against
the oracle models (bit-exact integers: step lists, block tables, slots, refcounts, free
counts), on random workloads that exercise chunking, the budget, recompute preemption and
prefix sharing."""
import numpy as np
import pytest

from continuous_batching_gb300 import binding as bd
from oracle import allocator as al
from oracle import scheduler as sc


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def _compare_state(cpp: bd.Scheduler, ref: sc.SchedulerModel):
    assert cpp.counts() == (len(ref.waiting), len(ref.running), ref.preemptions)
    assert cpp.allocator.num_free == ref.cache.alloc.num_free
    for q in ref.running:
        assert cpp.allocator.table(q) == ref.table(q)
        s = ref.seqs[q]
        assert cpp.seq(q) == (s.n_tokens, s.num_computed, s.generated)
    cpp.allocator.check_consistent()
    ref.cache.check_consistent()


@pytest.mark.parametrize("seed,num_blocks,bs,chunk,budget,share", [
    (0, 64, 16, 64, 256, False),
    (1, 24, 8, 24, 48, False),          # tight pool: preemption
    (2, 40, 8, 16, 40, True),           # prefix groups
    (3, 18, 4, 8, 20, True),            # tight pool + prefix groups
    (4, 200, 16, 512, 2048, True),      # the engine's chunk 512 / budget 2048 settings
])
def test_scheduler_matches_oracle_event_by_event(seed, num_blocks, bs, chunk, budget, share):
    rng = np.random.default_rng(seed)
    cpp = bd.Scheduler(num_blocks, bs, chunk, budget)
    ref = sc.SchedulerModel(num_blocks, bs, chunk, budget)
    next_id = 0
    leaders = []
    total_steps = 0
    for _ in range(400):
        # arrivals
        for _ in range(int(rng.integers(0, 3))):
            prompt = int(rng.integers(1, 5 * bs))
            max_new = int(rng.integers(1, 3 * bs))
            leader = None
            if share and leaders and rng.random() < 0.5:
                leader, prompt = leaders[int(rng.integers(0, len(leaders)))]
            # a request must fit the pool on its own, or it would wait forever
            if (prompt + max_new - 1 + bs - 1) // bs > num_blocks // 2:
                continue
            cpp.add(next_id, prompt, max_new, leader)
            ref.add(next_id, prompt, max_new, leader)
            if share and leader is None:
                leaders.append((next_id, prompt))
            next_id += 1
        got = cpp.step()
        want = ref.step()
        assert got == want
        for q, n, ctx in want:
            assert cpp.allocator.slots(q, ctx - n, n) == ref.slots(q, ctx - n, n)
        assert cpp.commit() == ref.commit()
        _compare_state(cpp, ref)
        total_steps += 1
    # drain
    for _ in range(20000):
        if ref.idle():
            break
        assert cpp.step() == ref.step()
        assert cpp.commit() == ref.commit()
    _compare_state(cpp, ref)
    assert ref.idle() and cpp.counts()[:2] == (0, 0)
    assert cpp.allocator.num_free == num_blocks
    if seed in (1, 3):
        assert ref.preemptions > 0


def test_step_feeds_build_step_like_the_oracle():
    cpp = bd.Scheduler(64, 16, 64, 256)
    ref = sc.SchedulerModel(64, 16, 64, 256)
    for i, (p, m) in enumerate([(40, 3), (5, 2), (130, 2), (17, 4)]):
        cpp.add(i, p, m)
        ref.add(i, p, m)
    for _ in range(6):
        st = cpp.step()
        assert st == ref.step()
        if st:
            seqs, n_new, ctx = (np.array(x, np.int32) for x in zip(*st))
            cu, slots, table = cpp.allocator.build_step(seqs, ctx, n_new, max_blocks=16)
            assert cu.tolist() == [0] + np.cumsum(n_new).tolist()
            want = sum((ref.slots(q, c - n, n) for q, n, c in st), [])
            assert slots.tolist() == want
            for i, q in enumerate(seqs):
                t = ref.table(int(q))
                nb = (int(ctx[i]) + 15) // 16
                assert table[i, :nb].tolist() == t[:nb]
                assert all(x == -1 for x in table[i, nb:])
        cpp.commit()
        ref.commit()


def test_trim_fork_cow_match_the_oracle():
    rng = np.random.default_rng(7)
    nb, bs = 48, 8
    cpp = bd.Allocator(nb, bs)
    ref = al.PagedCacheModel(nb, bs)
    lengths = {}
    next_id = 0
    for _ in range(3000):
        op = rng.integers(0, 6)
        live = sorted(lengths)
        try:
            if op == 0 or not live:
                n = int(rng.integers(1, 60))
                ref.admit(next_id, n)
                cpp.admit(next_id, n)
                lengths[next_id] = n
                next_id += 1
            elif op == 1:
                q = live[int(rng.integers(0, len(live)))]
                n = int(rng.integers(0, lengths[q] + 1))
                ref.trim(q, n)
                cpp.trim(q, n)
                lengths[q] = n
            elif op == 2:
                q = live[int(rng.integers(0, len(live)))]
                ref.fork(q, next_id)
                cpp.fork(q, next_id)
                lengths[next_id] = lengths[q]
                next_id += 1
            elif op == 3:
                q = live[int(rng.integers(0, len(live)))]
                n = lengths[q] + int(rng.integers(1, 20))
                ref.ensure_capacity(q, n)
                cpp.ensure_capacity(q, n)
                start = lengths[q]
                lengths[q] = n
                # make the positions about to be written private, copy-on-write
                s0 = max(0, start - int(rng.integers(0, 10)))
                want = ref.cow(q, s0, n - s0)       # the oracle first: it raises on exhaustion
                assert cpp.cow(q, s0, n - s0) == want
                assert cpp.slots(q, s0, n - s0) == ref.slots(q, s0, n - s0)
            elif op == 4:
                q = live[int(rng.integers(0, len(live)))]
                ref.free_seq(q)
                cpp.free_seq(q)
                del lengths[q]
            else:
                q = live[int(rng.integers(0, len(live)))]
                s0 = int(rng.integers(0, max(lengths[q], 1)))
                n = int(rng.integers(0, max(lengths[q] - s0, 0) + 1))
                want = ref.cow(q, s0, n)
                assert cpp.cow(q, s0, n) == want
        except al.PoolExhausted:
            with pytest.raises(bd.PoolExhausted):
                if op == 0:
                    cpp.admit(next_id, n)
                elif op == 3:
                    cpp.ensure_capacity(q, n) if lengths[q] < n else cpp.cow(q, s0, n - s0)
                else:
                    cpp.cow(q, s0, n)
        assert cpp.num_free == ref.alloc.num_free
        for q in lengths:
            assert cpp.table(q) == ref.tables[q]
        cpp.check_consistent()
        ref.check_consistent()
    for q in list(lengths):
        cpp.free_seq(q)
        ref.free_seq(q)
    assert cpp.num_free == nb and ref.alloc.num_free == nb
