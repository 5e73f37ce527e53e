"""Seeded synthetic inputs for one flat ragged paged-attention step.

This module only draws random numbers and lays out input structures (context
lengths, query-row counts, block tables, bf16 bit patterns).  It holds none of
the attention arithmetic, the slot mapping or the allocator logic: the CPU
oracle and the CUDA path each implement those on their own and both consume
the arrays produced here.

The workloads stand in for the ones the "P3: native paged-KV
continuous-batching sampler" page describes (heavy-tailed prover rollout
lengths, "Why"; chunk 512 / budget 2048 engine settings, "GPU validation
plan"; G samples sharing one prompt, "Design / engine.py, Prefix sharing").
No dataset is read: every value is i.i.d. N(0, 1) rounded to bf16, every
length is drawn from the stated distribution with ``numpy.random.default_rng``.

Layouts (row-major, all little-endian):
  q          uint16 (bf16 bits) [T, Hq, D]
  k_new/v_new uint16 (bf16 bits) [T, Hkv, D]
  k_pool/v_pool uint16 (bf16 bits) [num_blocks, block_size, Hkv, D]
  block_table int32 [B, max_blocks], unused entries -1
  cu_seqlens_q int32 [B + 1], ctx_lens int32 [B]
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = ["Step", "CONFIG_NAMES", "make_config", "make_step", "subset", "f32_to_bf16_bits",
           "random_bf16"]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the 16-bit patterns.

    Input generation only (the values drawn are N(0,1), never NaN)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def random_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """i.i.d. N(0,1) values rounded to bf16, drawn in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclass
class Step:
    """One synthetic ragged step: metadata plus bf16 bit patterns."""
    name: str
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    ctx_lens: np.ndarray          # int32 [B], includes this step's tokens
    n_q: np.ndarray               # int32 [B], query rows (new tokens) per sequence
    cu_seqlens_q: np.ndarray      # int32 [B+1]
    block_table: np.ndarray       # int32 [B, max_blocks], -1 padded
    q: np.ndarray                 # uint16 [T, Hq, D]
    k_new: np.ndarray             # uint16 [T, Hkv, D]
    v_new: np.ndarray             # uint16 [T, Hkv, D]
    k_pool: Optional[np.ndarray] = None   # uint16 [num_blocks, bs, Hkv, D]
    v_pool: Optional[np.ndarray] = None
    seed: int = 0
    shared_blocks: int = 0        # blocks referenced by more than one table (prefix sharing)
    notes: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def kv_tokens(self) -> int:
        """Logical K/V rows the step reads (sum of context lengths)."""
        return int(self.ctx_lens.astype(np.int64).sum())


CONFIG_NAMES = ("tiny", "decode", "mixed", "longtail", "prefix", "long16k")


def _blocks_for(ctx: np.ndarray, bs: int) -> np.ndarray:
    return (ctx.astype(np.int64) + bs - 1) // bs


def _perm_tables(rng, nblk_per_seq: np.ndarray, num_blocks: int) -> np.ndarray:
    """Tables whose entries are consecutive slices of one seeded permutation of the pool."""
    perm = rng.permutation(num_blocks).astype(np.int32)
    B = len(nblk_per_seq)
    mb = int(nblk_per_seq.max()) if B else 1
    table = np.full((B, max(mb, 1)), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(nblk_per_seq):
        n = int(n)
        table[i, :n] = perm[off:off + n]
        off += n
    return table


def _finish(name, rng, Hq, Hkv, D, bs, num_blocks, ctx, n_q, table, with_pool, seed,
            shared_blocks=0, notes=None) -> Step:
    ctx = np.asarray(ctx, dtype=np.int32)
    n_q = np.asarray(n_q, dtype=np.int32)
    cu = np.zeros(len(ctx) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(n_q)
    T = int(cu[-1])
    q = random_bf16(rng, (T, Hq, D))
    k_new = random_bf16(rng, (T, Hkv, D))
    v_new = random_bf16(rng, (T, Hkv, D))
    st = Step(name=name, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, num_blocks=int(num_blocks),
              ctx_lens=ctx, n_q=n_q, cu_seqlens_q=cu, block_table=table, q=q,
              k_new=k_new, v_new=v_new, seed=seed, shared_blocks=shared_blocks,
              notes=notes or {})
    if with_pool:
        st.k_pool = random_bf16(rng, (num_blocks, bs, Hkv, D))
        st.v_pool = random_bf16(rng, (num_blocks, bs, Hkv, D))
    return st


def make_config(name: str, with_pool: bool = True, seed: Optional[int] = None) -> Step:
    """Build one of the five named workloads.

    tiny     Hq 4, Hkv 2, D 64, bs 16, 32-block pool, ctx {17,40,64,100}, one decode row each.
    decode   Hq 32, Hkv 8, D 128, bs 16, 64 decode rows, ctx ~ lognormal(ln 2048, 1) clipped
             to [16, 16384], pool = sum(ceil(ctx/16)) blocks, permuted tables.
    mixed    Hq 32, Hkv 8, D 128, bs 16: 48 decode rows (ctx ~ lognormal(ln 3000, 1), clipped
             to [16, 16384]) plus 4 chunked-prefill segments of 512 rows at prior offsets
             {0, 512, 4096, 9000}; T = 2096.
    longtail Hq 64, Hkv 8, D 128, bs 32, 128 decode rows: 13 with ctx ~ U[16k, 40k] at seeded
             positions, 115 with ctx ~ U[1k, 4k].
    prefix   Hq 32, Hkv 8, D 128, bs 16: 16 prompts of 1024 tokens x 8 samples; each sample's
             table starts with its prompt's 64 full blocks (shared by 8 tables) followed by
             its own blocks for a U[1, 3000]-token continuation; 128 decode rows.
    long16k  Hq 32, Hkv 8, D 128, bs 16: 32 decode rows, every one at ctx 16,384 (the cap of
             the decode batch's lengths), permuted tables.
    """
    seeds = {"tiny": 0, "decode": 1, "mixed": 2, "longtail": 3, "prefix": 4, "long16k": 5}
    if name not in seeds:
        raise KeyError(f"unknown workload {name!r}; expected one of {CONFIG_NAMES}")
    seed = seeds[name] if seed is None else seed
    rng = np.random.default_rng(seed)
    if name == "tiny":
        Hq, Hkv, D, bs, nb = 4, 2, 64, 16, 32
        ctx = np.array([17, 40, 64, 100], dtype=np.int32)
        table = _perm_tables(rng, _blocks_for(ctx, bs), nb)
        return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, np.ones(4, np.int32), table,
                       with_pool, seed)
    if name == "decode":
        Hq, Hkv, D, bs, B = 32, 8, 128, 16, 64
        ctx = np.clip(np.rint(rng.lognormal(np.log(2048.0), 1.0, B)), 16, 16384).astype(np.int32)
        nblk = _blocks_for(ctx, bs)
        nb = int(nblk.sum())
        table = _perm_tables(rng, nblk, nb)
        return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, np.ones(B, np.int32), table,
                       with_pool, seed)
    if name == "mixed":
        Hq, Hkv, D, bs = 32, 8, 128, 16
        dec = np.clip(np.rint(rng.lognormal(np.log(3000.0), 1.0, 48)), 16, 16384).astype(np.int32)
        offs = np.array([0, 512, 4096, 9000], dtype=np.int32)
        ctx = np.concatenate([dec, offs + 512]).astype(np.int32)
        n_q = np.concatenate([np.ones(48, np.int32), np.full(4, 512, np.int32)])
        nblk = _blocks_for(ctx, bs)
        nb = int(nblk.sum())
        table = _perm_tables(rng, nblk, nb)
        return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, n_q, table, with_pool, seed,
                       notes={"prefill_offsets": offs.tolist()})
    if name == "long16k":
        Hq, Hkv, D, bs, B = 32, 8, 128, 16, 32
        ctx = np.full(B, 16384, dtype=np.int32)
        nblk = _blocks_for(ctx, bs)
        nb = int(nblk.sum())
        table = _perm_tables(rng, nblk, nb)
        return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, np.ones(B, np.int32), table,
                       with_pool, seed)
    if name == "longtail":
        Hq, Hkv, D, bs, B = 64, 8, 128, 32, 128
        n_long = int(round(0.1 * B))
        long_pos = np.sort(rng.choice(B, size=n_long, replace=False))
        ctx = rng.integers(1024, 4096, size=B, endpoint=True).astype(np.int32)
        ctx[long_pos] = rng.integers(16384, 40960, size=n_long, endpoint=True).astype(np.int32)
        nblk = _blocks_for(ctx, bs)
        nb = int(nblk.sum())
        table = _perm_tables(rng, nblk, nb)
        return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, np.ones(B, np.int32), table,
                       with_pool, seed, notes={"long_positions": long_pos.tolist()})
    # prefix
    return make_prefix_step(32, 8, 128, 16, prompts=16, samples=8, prompt_tokens=1024,
                            cont_max=3000, seed=seed, with_pool=with_pool, rng=rng)


def make_prefix_step(Hq: int, Hkv: int, D: int, block_size: int, prompts: int, samples: int,
                     prompt_tokens: int, cont_max: int, seed: int, with_pool: bool = True,
                     rng: Optional[np.random.Generator] = None, name: str = "prefix") -> Step:
    """Decode rows of `prompts` x `samples` sequences: each sample's table starts with its
    prompt's prompt_tokens // block_size full blocks (shared by the prompt's `samples` tables)
    followed by its own blocks for a U[1, cont_max]-token continuation (ctx = prompt_tokens +
    continuation); one decode row each, blocks a seeded permutation of the pool."""
    rng = np.random.default_rng(seed) if rng is None else rng
    bs, P, G = block_size, prompts, samples
    shared_per = prompt_tokens // bs
    cont = rng.integers(1, cont_max, size=P * G, endpoint=True).astype(np.int32)
    ctx = (prompt_tokens + cont).astype(np.int32)
    own = _blocks_for(ctx, bs) - shared_per
    nb = int(P * shared_per + own.sum())
    perm = rng.permutation(nb).astype(np.int32)
    mb = int(shared_per + own.max())
    table = np.full((P * G, mb), -1, dtype=np.int32)
    off = P * shared_per
    for p in range(P):
        shared = perm[p * shared_per:(p + 1) * shared_per]
        for g in range(G):
            i = p * G + g
            n = int(own[i])
            table[i, :shared_per] = shared
            table[i, shared_per:shared_per + n] = perm[off:off + n]
            off += n
    return _finish(name, rng, Hq, Hkv, D, bs, nb, ctx, np.ones(P * G, np.int32), table,
                   with_pool, seed, shared_blocks=P * shared_per,
                   notes={"prompts": P, "samples": G, "prompt_tokens": prompt_tokens})


def make_step(Hq: int, Hkv: int, D: int, block_size: int, ctx_lens, n_q, seed: int,
              num_blocks: Optional[int] = None, table: str = "perm",
              with_pool: bool = True, name: str = "custom") -> Step:
    """A custom step for tests: given context lengths and query-row counts per sequence.

    table="perm" draws a seeded permutation of the pool, "contig" assigns blocks in order.
    num_blocks defaults to exactly the blocks the tables need."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    n_q = np.asarray(n_q, dtype=np.int32)
    if np.any(n_q > ctx) or np.any(ctx < 1) or np.any(n_q < 0):
        raise ValueError("need 1 <= ctx and 0 <= n_q <= ctx")
    nblk = _blocks_for(ctx, block_size)
    need = int(nblk.sum())
    nb = need if num_blocks is None else int(num_blocks)
    if nb < need:
        raise ValueError("pool too small for the requested tables")
    if table == "perm":
        tab = _perm_tables(rng, nblk, nb)
    elif table == "contig":
        mb = int(nblk.max()) if len(nblk) else 1
        tab = np.full((len(ctx), max(mb, 1)), -1, dtype=np.int32)
        off = 0
        for i, n in enumerate(nblk):
            tab[i, :int(n)] = np.arange(off, off + int(n), dtype=np.int32)
            off += int(n)
    else:
        raise ValueError(table)
    return _finish(name, rng, Hq, Hkv, D, block_size, nb, ctx, n_q, tab, with_pool, seed)


def subset(step: Step, idx, k_pool=None, v_pool=None, name: str = "subset"):
    """A step made of sequences ``idx`` of ``step`` (same tables, rows and pool).

    Returns (Step, rows) where rows[j] are the token indices of sequence idx[j] in ``step``."""
    idx = [int(i) for i in idx]
    rows = [np.arange(step.cu_seqlens_q[s], step.cu_seqlens_q[s + 1]) for s in idx]
    n_q = np.array([len(r) for r in rows], np.int32)
    cu = np.zeros(len(idx) + 1, np.int32)
    cu[1:] = np.cumsum(n_q)
    allr = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    mb = step.block_table.shape[1]
    sub = Step(name=name, Hq=step.Hq, Hkv=step.Hkv, D=step.D, block_size=step.block_size,
               num_blocks=step.num_blocks, ctx_lens=step.ctx_lens[idx].copy(), n_q=n_q,
               cu_seqlens_q=cu, block_table=step.block_table[idx].reshape(len(idx), mb).copy(),
               q=step.q[allr], k_new=step.k_new[allr], v_new=step.v_new[allr],
               k_pool=step.k_pool if k_pool is None else k_pool,
               v_pool=step.v_pool if v_pool is None else v_pool, seed=step.seed)
    return sub, rows
