"""Paged KV store and causal attention, written as plain fp64 definitions.

Test infrastructure only (see the package docstring): the product never imports this.

Citations name the page and section they follow:
  [P3-paged]  "P3: native paged-KV continuous-batching sampler", Design / paged.py
  [P3-engine] same page, Design / engine.py (scheduler: flat ragged step, decodes + chunks)
  [P3-review] same page, Review ("Pool guard off by one", mutants list in Evidence item 5)
  [P3-tp]     same page, Tensor parallelism / Design (GQA "blocked map q_head // group")
  [MLX-v1]    "Optional paged KV cache (vLLM-style) — v1 design", Design (takeAxis gather,
              transpose, reshape, slice to offset) and Implementation order (bit-exact gate)

Readings where the pages leave a step open (each also listed in the design notes):
  * ctx_lens[s] counts this step's tokens: the step first writes its new K/V, then every
    query row attends ([P3-paged]: the attention seam "write new K/V, return [T, H, D]").
  * Query row i of sequence s (0 <= i < n_q) sits at absolute position ctx - n_q + i and
    attends keys 0..position inclusive (causal at an offset; [P3-engine] chunked prefill
    and decode share one flat ragged step).
  * The softmax scale is 1/sqrt(D) (the torch SDPA default that the per-row mode uses).
  * A slot < 0 means "no write" for that token.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

__all__ = ["bf16_to_f64", "slot_mapping", "kv_write", "gather", "row_positions",
           "attention", "attention_rows", "step", "kv_bytes_per_token",
           "blocks_needed", "cached_tokens"]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def slot_mapping(block_table: np.ndarray, cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray,
                 block_size: int) -> np.ndarray:
    """Physical slot of every new token of the step.  [P3-paged] "copy-free append
    (write scatters into (block, offset) in place)"; the mutant list in [P3-review]
    ("slot mapping ignores block offset") fixes that the offset inside the block counts.

    Token i of sequence s is at position p = ctx - n_q + i; its slot is
    table[s][p // block_size] * block_size + p % block_size.  Returns int64 [T]."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    T = int(cu[-1])
    out = np.empty(T, dtype=np.int64)
    for s in range(len(ctx)):
        n = int(cu[s + 1] - cu[s])
        for i in range(n):
            p = int(ctx[s]) - n + i
            blk = int(block_table[s, p // block_size])
            out[cu[s] + i] = blk * block_size + p % block_size
    return out


def kv_write(pool: np.ndarray, new: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Return a copy of ``pool`` [num_blocks, bs, Hkv, D] with row ``new[t]`` placed at
    ``slots[t]`` (skipped when slots[t] < 0).  Bytes are copied unchanged ([P3-paged])."""
    out = np.array(pool, copy=True)
    nb, bs = out.shape[0], out.shape[1]
    flat = out.reshape(nb * bs, *out.shape[2:])
    for t, s in enumerate(np.asarray(slots, dtype=np.int64)):
        if s < 0:
            continue
        if s >= nb * bs:
            raise IndexError(f"slot {s} outside a pool of {nb * bs} slots")
        flat[s] = new[t]
    return out


def gather(pool: np.ndarray, table_row: Sequence[int], ctx: int) -> np.ndarray:
    """Contiguous [Hkv, ctx, D] view of one sequence ([P3-paged] "gather() returns
    contiguous [1, Hkv, L, D]"; [MLX-v1] take whole blocks along axis 0, move the head
    axis first, merge block and offset axes, slice to the offset).  Same dtype as pool."""
    bs = pool.shape[1]
    nblk = (ctx + bs - 1) // bs
    blocks = pool[np.asarray(table_row[:nblk], dtype=np.int64)]      # [nblk, bs, Hkv, D]
    seq = blocks.reshape(nblk * bs, pool.shape[2], pool.shape[3])     # [nblk*bs, Hkv, D]
    return np.ascontiguousarray(seq[:ctx].transpose(1, 0, 2))          # [Hkv, ctx, D]


def row_positions(cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray) -> tuple:
    """(sequence index, absolute position) of every query row of the step."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    T = int(cu[-1])
    seq = np.empty(T, dtype=np.int64)
    pos = np.empty(T, dtype=np.int64)
    for s in range(len(ctx)):
        n = int(cu[s + 1] - cu[s])
        seq[cu[s]:cu[s + 1]] = s
        pos[cu[s]:cu[s + 1]] = ctx[s] - n + np.arange(n)
    return seq, pos


def _attend_sequence(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray, pos: np.ndarray,
                     Hq: int, scale: float) -> np.ndarray:
    """Causal softmax attention for some rows of one sequence, all fp64.

    q_rows [n, Hq, D]; K, V [Hkv, L, D]; pos [n] absolute positions.  Row r, head h reads
    kv head h // (Hq // Hkv) ([P3-tp]) and keys 0..pos[r] inclusive."""
    Hkv, L, D = K.shape
    g = Hq // Hkv
    kv_of = np.arange(Hq) // g
    out = np.empty((q_rows.shape[0], Hq, D), dtype=np.float64)
    for r in range(q_rows.shape[0]):
        n_keys = int(pos[r]) + 1
        Kh = K[kv_of, :n_keys, :]                 # [Hq, n_keys, D]
        Vh = V[kv_of, :n_keys, :]
        s = np.einsum("hd,hkd->hk", q_rows[r], Kh) * scale
        s = s - s.max(axis=1, keepdims=True)
        w = np.exp(s)
        w = w / w.sum(axis=1, keepdims=True)
        out[r] = np.einsum("hk,hkd->hd", w, Vh)
    return out


def attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_table: np.ndarray,
              cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray, Hq: int,
              scale: Optional[float] = None) -> np.ndarray:
    """fp64 output [T, Hq, D] of the step's attention over an already-written pool.

    Inputs are bf16 bit patterns (uint16) or floats; every sequence is gathered to a
    contiguous cache and each query row attends its own causal prefix ([P3-paged] 'row'
    mode semantics; [MLX-v1] the paged store is a storage-layout change only)."""
    rows = np.arange(int(np.asarray(cu_seqlens_q)[-1]))
    return attention_rows(q, k_pool, v_pool, block_table, cu_seqlens_q, ctx_lens, Hq, rows,
                          scale)


def _as_f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def attention_rows(q, k_pool, v_pool, block_table, cu_seqlens_q, ctx_lens, Hq: int,
                   rows, scale: Optional[float] = None) -> np.ndarray:
    """Like ``attention`` but only for the query rows listed in ``rows`` (token indices),
    so that full-size steps can be checked on a sample.  Returns [len(rows), Hq, D]."""
    rows = np.asarray(rows, dtype=np.int64)
    D = k_pool.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    seq_of, pos_of = row_positions(cu_seqlens_q, ctx_lens)
    out = np.empty((len(rows), Hq, D), dtype=np.float64)
    for s in np.unique(seq_of[rows]) if len(rows) else []:
        sel = np.nonzero(seq_of[rows] == s)[0]
        ctx = int(ctx_lens[s])
        K = _as_f64(gather(k_pool, block_table[s], ctx))
        V = _as_f64(gather(v_pool, block_table[s], ctx))
        qr = _as_f64(q[rows[sel]])
        out[sel] = _attend_sequence(qr, K, V, pos_of[rows[sel]], Hq, scale)
    return out


def step(q, k_new, v_new, k_pool, v_pool, block_table, cu_seqlens_q, ctx_lens, Hq: int,
         block_size: int, scale: Optional[float] = None):
    """The whole hot path as one definition: slots, KV write, then attention.

    Returns (slots int64 [T], k_pool_after, v_pool_after, out fp64 [T, Hq, D])."""
    slots = slot_mapping(block_table, cu_seqlens_q, ctx_lens, block_size)
    kp = kv_write(k_pool, k_new, slots)
    vp = kv_write(v_pool, v_new, slots)
    out = attention(q, kp, vp, block_table, cu_seqlens_q, ctx_lens, Hq, scale)
    return slots, kp, vp, out


# ---- memory accounting and sizing rules printed on the P3 page ------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int,
                       tp_degree: int = 1) -> int:
    """K and V bytes per cached token over all layers ([P3 page] Design / paged.py
    kv_bytes_per_token; Memory accounting: layers x 2 x kv-heads x head_dim x bytes,
    kv heads divided by the tensor-parallel degree)."""
    if kv_heads % tp_degree:
        raise ValueError("tp_degree must divide kv_heads")
    return layers * 2 * (kv_heads // tp_degree) * head_dim * dtype_bytes


def cached_tokens(prompt_len: int, max_new: int) -> int:
    """Tokens a finished request holds in the cache: the last sampled token is never fed
    back, so a request that ends with N tokens caches N - 1 ([P3-review], pool guard)."""
    return prompt_len + max_new - 1


def blocks_needed(n_tokens: int, block_size: int) -> int:
    """Blocks that cover n_tokens cached tokens."""
    return (n_tokens + block_size - 1) // block_size
