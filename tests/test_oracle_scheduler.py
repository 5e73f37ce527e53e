"""Pins for the reference scheduler and the allocator's rollback / copy-on-write model, against
what "P3: native paged-KV continuous-batching sampler" states (Design / engine.py: scheduler,
admit/evict, prefix sharing; Review: pool guard sweep, recompute preemption bill) and what
"Optional paged KV cache (vLLM-style) - v1 design" states for trim and block-level CoW."""
import numpy as np
import pytest

from oracle import allocator as al
from oracle import scheduler as sc


def run_to_end(m: sc.SchedulerModel, max_steps=100000):
    steps = []
    for _ in range(max_steps):
        if m.idle():
            return steps
        st = m.step()
        m.cache.check_consistent()
        m.commit()
        m.cache.check_consistent()
        steps.append(st)
    raise AssertionError("did not finish")


@pytest.mark.parametrize("prompt", range(1, 10))
@pytest.mark.parametrize("max_new", [1, 2, 3, 4, 5, 8, 9])
def test_pool_guard_sweep_exact_fit(prompt, max_new):
    """Review, "Pool guard off by one": a request ending with N tokens holds N - 1 in the
    cache; at block 4 a pool of exactly ceil((N - 1) / 4) blocks serves it, the peak use equals
    that, and the pool is fully free afterwards."""
    need = (prompt + max_new - 1 + 3) // 4
    m = sc.SchedulerModel(need, 4, chunk=512, budget=2048)
    m.add(0, prompt, max_new)
    peak = 0
    while not m.idle():
        m.step()
        peak = max(peak, need - m.cache.alloc.num_free)
        m.commit()
    assert m.seqs[0].generated == max_new
    assert peak == need and m.cache.alloc.num_free == need and m.preemptions == 0


def test_printed_example_prompt_3_plus_6_at_block_4_fits_two_blocks():
    m = sc.SchedulerModel(2, 4, chunk=512, budget=2048)
    m.add(0, 3, 6)
    run_to_end(m)
    assert m.seqs[0].generated == 6 and m.seqs[0].num_computed == 8


def test_decodes_first_chunked_prefill_and_budget():
    m = sc.SchedulerModel(64, 16, chunk=32, budget=48)
    m.add(0, 5, 4)
    st = m.step()
    assert st == [(0, 5, 5)]
    m.commit()
    m.add(1, 100, 2)                         # a long prompt arrives
    st = m.step()
    assert st[0] == (0, 1, 6)                # the decode first
    assert st[1] == (1, 32, 32)              # then a chunk of at most `chunk`
    assert sum(n for _, n, _ in st) <= 48
    m.commit()
    for _ in range(3):
        st = m.step()
        assert st[0][0] == 0 and st[0][1] == 1 or st[0][0] == 1
        assert all(n <= 32 for _, n, _ in st) and sum(n for _, n, _ in st) <= 48
        m.commit()


def test_every_step_respects_chunk_budget_and_order_on_random_load():
    rng = np.random.default_rng(5)
    m = sc.SchedulerModel(40, 8, chunk=24, budget=40)
    for i in range(30):
        m.add(i, int(rng.integers(1, 60)), int(rng.integers(1, 20)))
    for _ in range(5000):
        if m.idle():
            break
        before = {q: m._remaining(m.seqs[q]) for q in m.running}
        st = m.step()
        assert sum(n for _, n, _ in st) <= 40 and all(1 <= n <= 24 for _, n, _ in st)
        # decodes among the sequences running before the step come first
        kinds = [before.get(q) == 1 for q, _, _ in st if q in before]
        assert kinds == sorted(kinds, reverse=True)
        for q, n, ctx in st:
            assert m.cache.slots(q, ctx - n, n)          # writes land in private blocks
        m.commit()
        m.cache.check_consistent()
    assert m.idle() and m.cache.alloc.num_free == 40
    assert all(m.seqs[i].generated == m.seqs[i].max_new for i in range(30))


def test_recompute_preemption_takes_the_youngest_and_keeps_results():
    """Admit/evict: on exhaustion the youngest unscheduled running sequence is preempted by
    recompute. Review: 1 long decoder + 6 arrivals of 24 prompt / 40 new tokens at block 4 on
    a small pool preempt repeatedly and spend more forward tokens than the minimum."""
    m = sc.SchedulerModel(30, 4, chunk=512, budget=2048)
    m.add(100, 8, 60)
    m.step()
    m.commit()
    for i in range(6):
        m.add(i, 24, 40)
    forward = 8
    victims = []
    while not m.idle():
        running = list(m.running)
        stamps = {q: m.seqs[q].stamp for q in running}
        n_before = m.preemptions
        st = m.step()
        forward += sum(n for _, n, _ in st)
        if m.preemptions > n_before:
            gone = [q for q in running if q not in m.running]
            # each victim was the youngest among the running ones not scheduled
            scheduled = {q for q, _, _ in st}
            for v in gone:
                assert all(stamps[v] >= stamps[q] for q in running
                           if q not in scheduled and q not in gone or q == v)
            victims += gone
        m.commit()
    assert m.preemptions > 0 and victims
    minimal = (8 + 60 - 1) + 6 * (24 + 40 - 1)
    assert forward > minimal
    assert all(m.seqs[i].generated == 40 for i in range(6)) and m.seqs[100].generated == 60
    assert m.cache.alloc.num_free == 30


def test_prefix_followers_share_full_blocks_and_recompute_last_prompt_token():
    """Prefix sharing: followers adopt the leader's leading full blocks, defer while the
    leader computes them, and always recompute their last prompt token."""
    bs, P = 8, 33                       # (33 - 1) // 8 = 4 shared blocks, 32 tokens
    m = sc.SchedulerModel(64, bs, chunk=16, budget=64)
    m.add(0, P, 3)
    for f in (1, 2, 3):
        m.add(f, P, 3, leader=0)
    st = m.step()
    assert [q for q, _, _ in st] == [0]          # followers defer: the leader has 16 of 32
    m.commit()
    st = m.step()                                # leader reaches 32: followers still wait
    assert [q for q, _, _ in st] == [0]
    m.commit()
    st = m.step()
    assert {q for q, _, _ in st} == {0, 1, 2, 3}
    for q, n, ctx in st:
        if q != 0:
            assert (n, ctx) == (1, 33)           # only the last prompt token is recomputed
            assert m.table(q)[:4] == m.table(0)[:4]
    for b in m.table(0)[:4]:
        assert m.cache.alloc.ref[b] == 4
    m.commit()
    run_to_end(m)
    assert m.cache.alloc.num_free == 64


def test_follower_of_a_finished_leader_is_admitted_without_sharing():
    m = sc.SchedulerModel(16, 4, chunk=64, budget=64)
    m.add(0, 9, 1)
    m.step()
    m.commit()                                   # the leader finishes at once
    m.add(1, 9, 1, leader=0)
    st = m.step()
    assert st == [(1, 9, 9)]


def test_trim_frees_tail_last_first_and_regrowth_reuses_them():
    m = al.PagedCacheModel(8, 4)
    m.admit(0, 16)                               # blocks 0..3
    m.trim(0, 5)                                 # keep 2 blocks
    assert m.tables[0] == [0, 1] and m.alloc.num_free == 6
    m.ensure_capacity(0, 16)
    assert m.tables[0] == [0, 1, 2, 3]           # the block nearest the kept part first
    with pytest.raises(ValueError):
        m.trim(0, 17)
    m.check_consistent()


def test_fork_and_copy_on_write():
    m = al.PagedCacheModel(8, 4)
    m.admit(0, 10)                               # blocks 0, 1, 2 (last one partial)
    m.fork(0, 1)
    assert m.tables[1] == [0, 1, 2] and all(m.alloc.ref[b] == 2 for b in (0, 1, 2))
    with pytest.raises(al.ReadOnlyBlock):
        m.slots(1, 10, 1)
    m.ensure_capacity(1, 13)                     # block 3 (private) for positions 12..
    pairs = m.cow(1, 10, 3)                      # positions 10..12: shared block 2 -> 4
    assert pairs == [(2, 4)] and m.tables[1] == [0, 1, 4, 3] and m.alloc.ref[2] == 1
    m.slots(1, 10, 3)
    m.check_consistent()
    # all or nothing: not enough blocks for two replacements
    n = al.PagedCacheModel(3, 4)
    n.admit(0, 8)
    n.fork(0, 1)
    with pytest.raises(al.PoolExhausted):
        n.cow(1, 0, 8)
    assert n.tables[1] == n.tables[0] and n.alloc.num_free == 1
    n.check_consistent()


def test_mutant_scheduler_without_decode_priority_is_caught():
    """A mutant that visits running sequences in admission order only (no decodes first) must
    fail the ordering check used above."""
    class NoPriority(sc.SchedulerModel):
        def step(self):
            keep = self._remaining
            self._remaining = lambda s: 2 if keep(s) >= 1 else keep(s)
            try:
                return super().step()
            finally:
                self._remaining = keep
    m = NoPriority(64, 16, chunk=32, budget=48)
    m.add(0, 100, 2)
    m.step()
    m.commit()
    m.add(1, 5, 4)
    m.step()
    m.commit()                                   # 1 finished its prompt: a decode now
    st = m.step()
    assert st[0][0] == 0                         # the mutant schedules the prefill first


# --------------------------------------------------------------- pins that kill mutants
# The P3 page's Evidence item 5 asks that planted mistakes be killed. Each pin below is a
# property the page states (Design / engine.py, Admit/evict and Prefix sharing); it passes on
# the model and fails on a mutant that breaks exactly that property.

def pin_preemption(model_cls):
    """Admit/evict: on exhaustion the youngest running sequence not yet scheduled is preempted
    by recompute (its blocks freed, num_computed = 0); the books balance after every step and
    the pool is fully free at the end, every request having produced all its tokens."""
    m = model_cls(30, 4, chunk=512, budget=2048)
    m.add(100, 8, 60)
    m.step()
    m.commit()
    for i in range(6):
        m.add(i, 24, 40)
    for _ in range(10000):
        if m.idle():
            break
        running = list(m.running)
        stamps = {q: m.seqs[q].stamp for q in running}
        n_before = m.preemptions
        try:
            st = m.step()
            m.cache.check_consistent()
        except Exception as e:                 # the model itself gave up
            raise AssertionError(f"step failed: {e!r}")
        scheduled = {q for q, _, _ in st}
        gone = [q for q in running if q not in m.running]
        assert len(gone) == m.preemptions - n_before
        for v in gone:
            # the victim was younger than every other sequence it could have been
            others = [q for q in running if q not in scheduled and q != v and q not in gone]
            assert all(stamps[v] > stamps[q] for q in others), "not the youngest"
            assert v not in m.cache.tables, "a preempted sequence keeps its blocks"
            assert m.seqs[v].num_computed == 0
        try:
            m.commit()
            m.cache.check_consistent()
        except Exception as e:
            raise AssertionError(f"commit failed: {e!r}")
    assert m.idle() and m.preemptions > 0
    assert m.cache.alloc.num_free == 30
    assert all(m.seqs[i].generated == 40 for i in range(6)) and m.seqs[100].generated == 60


def pin_prefix_sharing(model_cls, P, bs=8):
    """Prefix sharing: a follower adopts only leading FULL blocks of its leader, shares every
    full block before its last prompt token, and always recomputes that token: its first
    step starts at the first unshared position and ends at ctx == P with n >= 1. Its writes
    land in private blocks and the pool is free at the end."""
    m = model_cls(64, bs, chunk=16, budget=64)
    m.add(0, P, 3)
    for f in (1, 2, 3):
        m.add(f, P, 3, leader=0)
    first = {}
    for _ in range(1000):
        if m.idle():
            break
        try:
            st = m.step()
        except Exception as e:
            raise AssertionError(f"step failed: {e!r}")
        for q, n, ctx in st:
            if q in (1, 2, 3) and q not in first:
                assert 0 in m.cache.tables, "the leader finished before its followers ran"
                shared = [b for b in m.table(q) if m.cache.alloc.ref[b] > 1]
                k = len(shared)
                assert m.table(q)[:k] == m.table(0)[:k], "shared blocks are not the leader's"
                assert k * bs <= P - 1, "a shared block holds the last prompt token or is partial"
                assert (k + 1) * bs > P - 1, "a full block before the last token is not shared"
                assert n >= 1 and ctx - n == k * bs and ctx <= P, (q, n, ctx, k)
                first[q] = (n, ctx)
            try:
                m.slots(q, ctx - n, n)
            except Exception as e:
                raise AssertionError(f"write of sequence {q} refused: {e!r}")
        try:
            m.commit()
            m.cache.check_consistent()
        except Exception as e:
            raise AssertionError(f"commit failed: {e!r}")
    assert set(first) == {1, 2, 3}
    assert all(ctx == P or ctx < P for n, ctx in first.values())
    assert m.idle() and m.cache.alloc.num_free == 64


def pin_youngest_victim(model_cls):
    """Admit/evict, "preempt the youngest": A, B, C (admitted in that order) decode in lockstep
    until their next block is missing for all three. The visit serves A first (decodes in
    admission order); the candidates are then B and C, and C, the youngest, must go back to
    waiting while A and B both run."""
    m = model_cls(6, 4, chunk=512, budget=2048)
    for i in range(3):
        m.add(i, 4, 10)
    for _ in range(20):
        st = m.step()
        m.commit()
        if m.preemptions:
            break
    assert m.preemptions == 1, m.preemptions
    assert [q for q, _, _ in st] == [0, 1], st
    assert list(m.waiting) == [2] and m.running == [0, 1]


class _OldestVictim(sc.SchedulerModel):
    def _pick_victim(self, victims):
        return min(victims, key=lambda v: self.seqs[v].stamp)


class _PreemptKeepsBlocks(sc.SchedulerModel):
    def _preempt(self, q):
        self.running.remove(q)
        s = self.seqs[q]
        s.num_computed = 0
        s.stamp = -1
        self.waiting.appendleft(q)
        self.preemptions += 1


class _SharesPartialBlock(sc.SchedulerModel):
    def _shared_blocks(self, s):
        return (s.prompt_len + self.bs - 1) // self.bs


class _NoLastTokenRecompute(sc.SchedulerModel):
    def _shared_blocks(self, s):
        return s.prompt_len // self.bs


def test_pins_pass_on_the_model():
    pin_youngest_victim(sc.SchedulerModel)
    pin_preemption(sc.SchedulerModel)
    for P in (30, 32, 33, 9, 8):
        pin_prefix_sharing(sc.SchedulerModel, P)


@pytest.mark.parametrize("mutant,pin", [
    (_OldestVictim, lambda c: pin_youngest_victim(c)),
    (_PreemptKeepsBlocks, lambda c: pin_preemption(c)),
    (_SharesPartialBlock, lambda c: pin_prefix_sharing(c, 30)),
    (_NoLastTokenRecompute, lambda c: pin_prefix_sharing(c, 32)),
])
def test_scheduler_mutants_are_killed(mutant, pin):
    with pytest.raises(AssertionError):
        pin(mutant)
