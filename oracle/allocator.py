"""Reference model of the block allocator and per-sequence block tables.

Test infrastructure only (see the package docstring): the product never imports this.

Follows "P3: native paged-KV continuous-batching sampler", Design / paged.py:
  * BlockAllocator: a LIFO free list plus refcounts; freeing a block whose refcount is
    already 0 raises (a double free would hand one block to two sequences);
    check_consistent proves free + referenced == total with no duplicates.
  * PagedKVCache: ensure_capacity is all-or-nothing; slots() refuses a write into a block
    with refcount > 1 (read-only for everyone, the owner included).
  * Prefix sharing (Design / engine.py): a sequence adopts the leading FULL blocks of a
    running one.
and Evidence item 4 (books checked after every event against refcounts recomputed from
the live block tables).  The typed exhaustion error follows "Optional paged KV cache
(vLLM-style) — v1 design", Design (alloc throws PagedPoolExhausted: never silent
truncation).

Reading where the pages leave it open: the free stack starts so that the first alloc
returns block 0; free pushes on top, so the next alloc reuses the most recently freed
block.

Rollback and copy-on-write follow "Optional paged KV cache (vLLM-style) — v1 design":
  * trim(n) rewinds a sequence to n tokens and frees the now-unoccupied tail blocks (stale
    bytes past the offset are never read). Reading: tail blocks are freed from the last one
    backwards, so the block nearest the kept part is handed out first when the sequence
    grows again.
  * Block-level CoW sharing (refcounted block tables, fork-on-divergent-write): fork gives
    a new sequence every block of an existing one (refcounts up, partial last block
    included); before a write into positions that lie in blocks with refcount > 1, each such
    block is replaced by a fresh private block, and the (old, new) pairs are returned so the
    caller copies the old contents first. Reading: blocks are replaced in table order, all
    or nothing (if the pool cannot supply every replacement nothing changes).
"""
from __future__ import annotations

from typing import Dict, List, Optional


class PoolExhausted(Exception):
    """Not enough free blocks; nothing was changed."""


class DoubleFree(Exception):
    """Free of a block whose refcount is already 0."""


class ReadOnlyBlock(Exception):
    """A write would land in a block referenced by more than one table."""


class Inconsistent(AssertionError):
    """The books do not balance."""


class BlockAllocator:
    def __init__(self, num_blocks: int):
        if num_blocks < 0:
            raise ValueError("num_blocks < 0")
        self.num_blocks = num_blocks
        self.free_list: List[int] = list(range(num_blocks - 1, -1, -1))
        self.ref = [0] * num_blocks

    @property
    def num_free(self) -> int:
        return len(self.free_list)

    def alloc(self) -> int:
        if not self.free_list:
            raise PoolExhausted("pool exhausted")
        b = self.free_list.pop()
        self.ref[b] = 1
        return b

    def incref(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise Inconsistent(f"incref of free block {b}")
        self.ref[b] += 1

    def free(self, b: int) -> None:
        if self.ref[b] == 0:
            raise DoubleFree(f"block {b} already free")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free_list.append(b)

    def check_consistent(self, tables: Optional[Dict[int, List[int]]] = None) -> None:
        if len(set(self.free_list)) != len(self.free_list):
            raise Inconsistent("duplicate block on the free list")
        referenced = sum(1 for r in self.ref if r > 0)
        if referenced + len(self.free_list) != self.num_blocks:
            raise Inconsistent("free + referenced != total")
        for b in self.free_list:
            if self.ref[b] != 0:
                raise Inconsistent(f"block {b} on the free list has refcount {self.ref[b]}")
        if tables is not None:
            want = [0] * self.num_blocks
            for t in tables.values():
                for b in t:
                    want[b] += 1
            if want != self.ref:
                raise Inconsistent("refcounts differ from the live block tables")


class PagedCacheModel:
    """Per-sequence block tables on top of BlockAllocator."""

    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.alloc = BlockAllocator(num_blocks)
        self.tables: Dict[int, List[int]] = {}

    def _need(self, n_tokens: int) -> int:
        return (n_tokens + self.block_size - 1) // self.block_size

    def admit(self, seq: int, n_tokens: int, share_src: Optional[int] = None,
              n_shared: int = 0) -> None:
        """Create seq's table covering n_tokens; with share_src, adopt its first n_shared
        FULL blocks read-only.  All-or-nothing."""
        if seq in self.tables:
            raise ValueError(f"sequence {seq} already admitted")
        shared: List[int] = []
        if share_src is not None and n_shared > 0:
            src = self.tables[share_src]
            if n_shared > len(src) or n_shared * self.block_size > n_tokens:
                raise ValueError("can only share leading full blocks the new sequence covers")
            shared = src[:n_shared]
        need = self._need(n_tokens) - len(shared)
        if need > self.alloc.num_free:
            raise PoolExhausted(f"need {need}, have {self.alloc.num_free}")
        for b in shared:
            self.alloc.incref(b)
        self.tables[seq] = list(shared) + [self.alloc.alloc() for _ in range(max(need, 0))]

    def ensure_capacity(self, seq: int, n_tokens: int) -> None:
        t = self.tables[seq]
        need = self._need(n_tokens) - len(t)
        if need <= 0:
            return
        if need > self.alloc.num_free:
            raise PoolExhausted(f"need {need}, have {self.alloc.num_free}")
        t.extend(self.alloc.alloc() for _ in range(need))

    def free_seq(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.alloc.free(b)

    def slots(self, seq: int, start: int, n: int) -> List[int]:
        """Slots for positions start..start+n-1; refuses any block with refcount > 1."""
        t = self.tables[seq]
        out = []
        for p in range(start, start + n):
            j = p // self.block_size
            if j >= len(t):
                raise IndexError("position beyond the table's capacity")
            b = t[j]
            if self.alloc.ref[b] > 1:
                raise ReadOnlyBlock(f"block {b} is shared (refcount {self.alloc.ref[b]})")
            out.append(b * self.block_size + p % self.block_size)
        return out

    def trim(self, seq: int, n_tokens: int) -> None:
        """Rewind seq to n_tokens: keep the blocks that cover them, free the rest (last
        block first)."""
        t = self.tables[seq]
        keep = self._need(n_tokens)
        if n_tokens < 0 or keep > len(t):
            raise ValueError("trim beyond the table's capacity")
        for b in reversed(t[keep:]):
            self.alloc.free(b)
        del t[keep:]

    def fork(self, src: int, dst: int) -> None:
        """dst shares every block of src (copy-on-write)."""
        if dst in self.tables:
            raise ValueError(f"sequence {dst} already admitted")
        t = self.tables[src]
        for b in t:
            self.alloc.incref(b)
        self.tables[dst] = list(t)

    def cow(self, seq: int, start: int, n: int) -> List[tuple]:
        """Make the blocks holding positions start..start+n-1 private to seq. Returns the
        (old block, new block) pairs whose contents the caller must copy before writing."""
        t = self.tables[seq]
        if n <= 0:
            return []
        first, last = start // self.block_size, (start + n - 1) // self.block_size
        if start < 0 or last >= len(t):
            raise IndexError("position beyond the table's capacity")
        shared = [j for j in range(first, last + 1) if self.alloc.ref[t[j]] > 1]
        if len(shared) > self.alloc.num_free:
            raise PoolExhausted(f"need {len(shared)}, have {self.alloc.num_free}")
        pairs = []
        for j in shared:
            old = t[j]
            new = self.alloc.alloc()
            self.alloc.free(old)              # drops this table's reference only
            t[j] = new
            pairs.append((old, new))
        return pairs

    def check_consistent(self) -> None:
        self.alloc.check_consistent(self.tables)
