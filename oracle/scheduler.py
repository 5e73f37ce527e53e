"""Reference model of the step scheduler (host side of one flat ragged step).

Test infrastructure only (see the package docstring): the product never imports this.

Follows "P3: native paged-KV continuous-batching sampler", Design / engine.py:
  * Scheduler: every sequence is tokens + num_computed; a step schedules
    n_new = min(remaining, chunk_size, budget) per sequence; prefill, chunked prefill, decode
    and recompute after preemption are one path; a sequence samples when its scheduled
    tokens reach the end of its tokens; decodes are scheduled first; prefill chunks and
    decode tokens share one flat ragged step.
  * Admit/evict: FIFO admission if the whole current token list fits; on block exhaustion the
    youngest unscheduled running sequence is preempted by recompute (blocks freed,
    num_computed = 0, tokens kept).
  * Prefix sharing: a waiting sequence adopts the leading FULL blocks of a running sequence,
    defers while the leader is still computing them, and always recomputes its last prompt
    token.
and Review ("Pool guard off by one"): the last sampled token is never fed back, so a request
that ends with N tokens holds N - 1 in the cache.

Readings where the page is silent (each one is also listed in the design notes):
  S1  remaining = len(tokens) - num_computed; a decode is a running sequence with
      remaining == 1.
  S2  Running sequences are visited decodes first, then the others, each group in admission
      order; then waiting sequences are admitted FIFO while budget remains. Admission stops
      at the first waiting sequence that does not fit or defers.
  S3  A running sequence's blocks grow with ensure_capacity(num_computed + n_new). On
      exhaustion the youngest running sequence not yet scheduled in this step (not the one
      being scheduled) is preempted and the attempt repeats; with no such sequence left the
      sequence is skipped for this step and the visit goes on.
  S4  Admission allocates blocks for the whole current token list, all or nothing.
  S5  A preempted sequence goes back to the head of the waiting queue (the first victim of a
      step ends up behind the later ones, so the oldest victim is first).
  S6  A follower names a leader and a prompt length P; it shares (P - 1) // block_size full
      blocks. It defers while the leader is waiting or has computed fewer tokens than those
      blocks hold; if the leader has finished, it is admitted without sharing. A follower
      that shares starts with num_computed = shared blocks * block_size.
  S7  After a step, each scheduled sequence adds its n_new to num_computed; if that reaches
      len(tokens) it samples one token: a sequence that reached max_new finishes (blocks
      freed), any other appends the token.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Optional, Tuple

from .allocator import PagedCacheModel, PoolExhausted


class SeqState:
    def __init__(self, seq: int, prompt_len: int, max_new: int, leader: Optional[int]):
        self.seq = seq
        self.n_tokens = prompt_len          # len(tokens): prompt + sampled so far
        self.prompt_len = prompt_len
        self.num_computed = 0
        self.max_new = max_new
        self.generated = 0
        self.leader = leader
        self.stamp = -1                     # admission order of the current residency


class SchedulerModel:
    def __init__(self, num_blocks: int, block_size: int, chunk: int, budget: int):
        self.cache = PagedCacheModel(num_blocks, block_size)
        self.bs = block_size
        self.chunk = chunk
        self.budget = budget
        self.seqs: Dict[int, SeqState] = {}
        self.waiting: deque = deque()
        self.running: List[int] = []        # admission order
        self.finished: List[int] = []
        self.preemptions = 0
        self._stamp = 0
        self._scheduled: List[Tuple[int, int]] = []

    # -------------------------------------------------------------- requests
    def add(self, seq: int, prompt_len: int, max_new: int, leader: Optional[int] = None):
        if seq in self.seqs or prompt_len < 1 or max_new < 1:
            raise ValueError("bad request")
        self.seqs[seq] = SeqState(seq, prompt_len, max_new, leader)
        self.waiting.append(seq)

    def _remaining(self, s: SeqState) -> int:
        return s.n_tokens - s.num_computed

    # -------------------------------------------------------------- one step
    def step(self) -> List[Tuple[int, int, int]]:
        """Returns [(seq, n_new, ctx)] in step order (ctx = num_computed + n_new)."""
        budget = self.budget
        done: set = set()
        out: List[Tuple[int, int]] = []
        order = [q for q in self.running if self._remaining(self.seqs[q]) == 1] + \
                [q for q in self.running if self._remaining(self.seqs[q]) > 1]
        for q in order:
            if budget == 0:
                break
            if q not in self.running:       # preempted earlier in this step
                continue
            s = self.seqs[q]
            n = min(self._remaining(s), self.chunk, budget)
            while True:
                try:
                    self.cache.ensure_capacity(q, s.num_computed + n)
                    ok = True
                    break
                except PoolExhausted:
                    victims = [v for v in self.running if v not in done and v != q]
                    if not victims:
                        ok = False
                        break
                    self._preempt(self._pick_victim(victims))
            if ok:
                out.append((q, n))
                done.add(q)
                budget -= n
        while self.waiting and budget > 0:
            q = self.waiting[0]
            s = self.seqs[q]
            n_shared = 0
            src = None
            if s.leader is not None and s.leader in self.seqs:
                lead = self.seqs[s.leader]
                share = self._shared_blocks(s)
                if s.leader in self.finished:
                    share = 0
                elif s.leader not in self.running or lead.num_computed < share * self.bs:
                    break                       # defers while the leader computes
                if share > 0:
                    n_shared, src = share, s.leader
            try:
                self.cache.admit(q, s.n_tokens, share_src=src, n_shared=n_shared)
            except PoolExhausted:
                break
            self.waiting.popleft()
            self.running.append(q)
            s.stamp = self._stamp
            self._stamp += 1
            s.num_computed = n_shared * self.bs
            n = min(self._remaining(s), self.chunk, budget)
            out.append((q, n))
            done.add(q)
            budget -= n
        self._scheduled = out
        return [(q, n, self.seqs[q].num_computed + n) for q, n in out]

    def _pick_victim(self, victims: List[int]) -> int:
        """S3: the youngest (latest admitted) of the candidates."""
        return max(victims, key=lambda v: self.seqs[v].stamp)

    def _shared_blocks(self, s: SeqState) -> int:
        """S6: the leading full blocks before the last prompt token, which is recomputed."""
        return (s.prompt_len - 1) // self.bs

    def _preempt(self, q: int) -> None:
        self.cache.free_seq(q)
        self.running.remove(q)
        s = self.seqs[q]
        s.num_computed = 0
        s.stamp = -1
        self.waiting.appendleft(q)
        self.preemptions += 1

    def commit(self) -> List[int]:
        """Applies the last step's results; returns the sequences that finished."""
        fin = []
        for q, n in self._scheduled:
            s = self.seqs[q]
            s.num_computed += n
            if s.num_computed == s.n_tokens:
                s.generated += 1
                if s.generated == s.max_new:
                    self.cache.free_seq(q)
                    self.running.remove(q)
                    self.finished.append(q)
                    fin.append(q)
                else:
                    s.n_tokens += 1
        self._scheduled = []
        return fin

    # -------------------------------------------------------------- views
    def slots(self, seq: int, start: int, n: int) -> List[int]:
        return self.cache.slots(seq, start, n)

    def table(self, seq: int) -> List[int]:
        return list(self.cache.tables[seq])

    def idle(self) -> bool:
        return not self.waiting and not self.running
