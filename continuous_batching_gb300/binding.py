"""Thin ctypes binding of libpagedattn (the C ABI declared in include/pagedattn.h).

Argument marshalling only: every step of the hot path runs in the library's kernels. Device
buffers are torch CUDA tensors (PyTorch supplies device memory and streams); host buffers are
numpy arrays. Statuses other than PA_OK raise ``PagedAttnError`` (or a subclass).

The library is loaded on first use from this package's directory; a missing library raises
``RuntimeError`` (there is no fallback path).
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional

import numpy as np

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedattn.so")

PA_OK, PA_ERR_INVALID, PA_ERR_SHAPE, PA_ERR_BOUNDS, PA_ERR_OOM, PA_ERR_READONLY, \
    PA_ERR_DOUBLE_FREE, PA_ERR_INCONSISTENT, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_STATE = range(11)
PA_DEVERR_BLOCK, PA_DEVERR_SLOT, PA_DEVERR_TIMEOUT, PA_DEVERR_META = 1, 2, 4, 8
PA_SPLIT_TOKENS = 2048
PA_TILE_KEYS = 128
PA_PLAN_CTAS = 152


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" if where else status_string(status))


class PoolExhausted(PagedAttnError):
    """PA_ERR_OOM: not enough free blocks; nothing changed."""


class DoubleFree(PagedAttnError):
    """PA_ERR_DOUBLE_FREE."""


class ReadOnlyBlock(PagedAttnError):
    """PA_ERR_READONLY: a write would land in a shared block."""


_ERRORS = {PA_ERR_OOM: PoolExhausted, PA_ERR_DOUBLE_FREE: DoubleFree,
           PA_ERR_READONLY: ReadOnlyBlock}


class Shape(C.Structure):
    _fields_ = [("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("block_size", C.c_int32), ("num_blocks", C.c_int32)]

    @classmethod
    def make(cls, Hq, Hkv, D, block_size, num_blocks) -> "Shape":
        return cls(int(Hq), int(Hkv), int(D), int(block_size), int(num_blocks))


class WorkItem(C.Structure):
    _fields_ = [("seq", C.c_int32), ("q_start", C.c_int32), ("n_q", C.c_int32),
                ("kv_head", C.c_int32), ("split", C.c_int32), ("n_tiles", C.c_int32),
                ("n_splits", C.c_int32), ("next", C.c_int32), ("kind", C.c_int32),
                ("tile0", C.c_int32)]


WORK_ITEM_DTYPE = np.dtype([(n, np.int32) for n, _ in WorkItem._fields_])
ITEM_INTS = len(WorkItem._fields_)          # int32 words per pa_work_item
PA_ITEM_PLAIN, PA_ITEM_GROUP, PA_ITEM_RESUME = 0, 1, 2

_lib = None
_lock = threading.Lock()
_i32p = C.POINTER(C.c_int32)
_vp = C.c_void_p


def _sig(lib, name, res, args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = args


def load() -> C.CDLL:
    """Loads libpagedattn.so (once); raises RuntimeError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() or "
                               "python -m continuous_batching_gb300.build")
        lib = C.CDLL(LIB_PATH)
        sp = C.POINTER(Shape)
        ap = C.c_void_p                  # pa_allocator*
        _sig(lib, "pa_abi_version", C.c_int32, [])
        _sig(lib, "pa_status_string", C.c_char_p, [C.c_int32])
        _sig(lib, "pa_last_cuda_error", C.c_int32, [])
        _sig(lib, "pa_device_sm_count", C.c_int32, [_i32p])
        _sig(lib, "pa_alloc_create", C.c_int32, [C.c_int32, C.c_int32, C.POINTER(ap)])
        _sig(lib, "pa_alloc_destroy", C.c_int32, [ap])
        _sig(lib, "pa_alloc_block", C.c_int32, [ap, _i32p])
        _sig(lib, "pa_alloc_incref", C.c_int32, [ap, C.c_int32])
        _sig(lib, "pa_alloc_free_block", C.c_int32, [ap, C.c_int32])
        _sig(lib, "pa_alloc_admit", C.c_int32, [ap, C.c_int32, C.c_int32, C.c_int32, C.c_int32])
        _sig(lib, "pa_alloc_ensure_capacity", C.c_int32, [ap, C.c_int32, C.c_int32])
        _sig(lib, "pa_alloc_free_seq", C.c_int32, [ap, C.c_int32])
        _sig(lib, "pa_alloc_check_consistent", C.c_int32, [ap])
        _sig(lib, "pa_alloc_num_free", C.c_int32, [ap])
        _sig(lib, "pa_alloc_refcount", C.c_int32, [ap, C.c_int32])
        _sig(lib, "pa_alloc_table", C.c_int32, [ap, C.c_int32, _i32p, C.c_int32, _i32p])
        _sig(lib, "pa_alloc_slots", C.c_int32, [ap, C.c_int32, C.c_int32, C.c_int32, _i32p])
        _sig(lib, "pa_alloc_build_step", C.c_int32,
             [ap, _i32p, _i32p, _i32p, C.c_int32, _i32p, _i32p, _i32p, C.c_int32])
        _sig(lib, "pa_alloc_trim", C.c_int32, [ap, C.c_int32, C.c_int32])
        _sig(lib, "pa_alloc_fork", C.c_int32, [ap, C.c_int32, C.c_int32])
        _sig(lib, "pa_alloc_cow", C.c_int32,
             [ap, C.c_int32, C.c_int32, C.c_int32, _i32p, C.c_int32, _i32p])
        sc = C.c_void_p                  # pa_scheduler*
        _sig(lib, "pa_sched_create", C.c_int32,
             [C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(sc)])
        _sig(lib, "pa_sched_destroy", C.c_int32, [sc])
        _sig(lib, "pa_sched_allocator", ap, [sc])
        _sig(lib, "pa_sched_add", C.c_int32, [sc, C.c_int32, C.c_int32, C.c_int32, C.c_int32])
        _sig(lib, "pa_sched_step", C.c_int32, [sc, _i32p, _i32p, _i32p, C.c_int32, _i32p])
        _sig(lib, "pa_sched_commit", C.c_int32, [sc, _i32p, C.c_int32, _i32p])
        _sig(lib, "pa_sched_counts", C.c_int32, [sc, _i32p, _i32p, C.POINTER(C.c_int64)])
        _sig(lib, "pa_sched_seq", C.c_int32, [sc, C.c_int32, _i32p, _i32p, _i32p])
        _sig(lib, "pa_compute_slots", C.c_int32,
             [sp, _i32p, C.c_int32, C.c_int32, _i32p, _i32p, _i32p])
        _sig(lib, "pa_plan_max_items", C.c_int64, [sp, C.c_int32, C.c_int32, C.c_int32])
        _sig(lib, "pa_plan_step", C.c_int32,
             [sp, C.c_int32, _i32p, _i32p, C.POINTER(WorkItem), C.c_int32, _i32p])
        _sig(lib, "pa_plan_max_items_shared", C.c_int64, [sp, C.c_int32, C.c_int32, C.c_int32])
        _sig(lib, "pa_plan_step_shared", C.c_int32,
             [sp, C.c_int32, _i32p, _i32p, _i32p, C.c_int32, C.POINTER(WorkItem), C.c_int32,
              _i32p])
        _sig(lib, "pa_workspace_bytes", C.c_size_t, [sp, C.c_int32, C.c_int32])
        _sig(lib, "pa_upload_block_table", C.c_int32,
             [sp, _i32p, _vp, C.c_int32, C.c_int32, _vp])
        _sig(lib, "paged_kv_write", C.c_int32,
             [_vp, _vp, _vp, C.c_int32, _vp, _vp, sp, _vp, _vp])
        _sig(lib, "paged_copy_blocks", C.c_int32, [_vp, C.c_int32, _vp, _vp, sp, _vp, _vp])
        _sig(lib, "paged_attention_step", C.c_int32,
             [_vp, _vp, _vp, _vp, C.c_int32, _vp, _vp, C.c_int32, C.c_int32, C.c_int32,
              _vp, C.c_int32, _vp, C.c_size_t, _vp, sp, _vp, _vp])
        _sig(lib, "paged_attention_step_wait_test", C.c_int32,
             [_vp, _vp, _vp, _vp, C.c_int32, _vp, _vp, C.c_int32, C.c_int32, C.c_int32,
              _vp, C.c_int32, _vp, C.c_size_t, _vp, sp, _vp, C.c_uint64, _vp])
        pp = C.c_void_p                  # pa_pipeline*
        _sig(lib, "pa_pipeline_create", C.c_int32,
             [sp, C.c_int32, C.c_int32, C.c_int32, C.c_int32, _vp, _vp, C.c_int32, C.c_float,
              C.c_float, C.POINTER(pp)])
        _sig(lib, "pa_pipeline_destroy", C.c_int32, [pp])
        _sig(lib, "pa_pipeline_meta_bytes", C.c_int64, [pp])
        _sig(lib, "pa_pipeline_submit", C.c_int32,
             [pp, _i32p, _i32p, _i32p, C.c_int32, _vp, _vp, _vp, _vp, _i32p])
        _sig(lib, "pa_pipeline_wait", C.c_int32, [pp, C.c_int32])
        _sig(lib, "pa_pipeline_device_error", C.c_int32, [pp, _i32p])
        _sig(lib, "paged_kv_write_fp8", C.c_int32,
             [_vp, _vp, _vp, C.c_int32, _vp, _vp, C.c_float, C.c_float, sp, _vp, _vp])
        _sig(lib, "paged_attention_step_fp8", C.c_int32,
             [_vp, _vp, _vp, _vp, C.c_int32, _vp, _vp, C.c_int32, C.c_int32, C.c_int32,
              _vp, C.c_int32, C.c_float, C.c_float, _vp, C.c_size_t, _vp, sp, _vp, _vp])
        _lib = lib
        return lib


def status_string(st: int) -> str:
    try:
        return load().pa_status_string(int(st)).decode()
    except RuntimeError:
        return f"status {st}"


def _check(st: int, where: str) -> None:
    if st != PA_OK:
        if st == PA_ERR_CUDA:
            raise PagedAttnError(st, f"{where} (cudaError {load().pa_last_cuda_error()})")
        raise _ERRORS.get(st, PagedAttnError)(st, where)


def _i32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _p32(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_i32p)


def _dev(t) -> Optional[int]:
    """Device address of a torch tensor (or None)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ------------------------------------------------------------------------ library info

def pa_abi_version() -> int:
    return int(load().pa_abi_version())


def pa_device_sm_count() -> int:
    n = C.c_int32()
    _check(load().pa_device_sm_count(C.byref(n)), "pa_device_sm_count")
    return int(n.value)


# ---------------------------------------------------------------------- host allocator

class Allocator:
    """A pa_allocator (LIFO blocks, refcounts, read-only shared prefix blocks): owned, or
    borrowed from a Scheduler (then the scheduler frees it)."""

    def __init__(self, num_blocks: int, block_size: int, _borrow=None):
        self._lib = load()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self._owned = _borrow is None
        if _borrow is not None:
            self._h = _borrow
            return
        h = C.c_void_p()
        _check(self._lib.pa_alloc_create(int(num_blocks), int(block_size), C.byref(h)),
               "pa_alloc_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) and getattr(self, "_owned", False):
            self._lib.pa_alloc_destroy(self._h)
        self._h = None

    __del__ = close

    def alloc(self) -> int:
        b = C.c_int32()
        _check(self._lib.pa_alloc_block(self._h, C.byref(b)), "pa_alloc_block")
        return int(b.value)

    def incref(self, b: int) -> None:
        _check(self._lib.pa_alloc_incref(self._h, int(b)), "pa_alloc_incref")

    def free(self, b: int) -> None:
        _check(self._lib.pa_alloc_free_block(self._h, int(b)), "pa_alloc_free_block")

    def admit(self, seq: int, n_tokens: int, share_src: Optional[int] = None,
              n_shared: int = 0) -> None:
        _check(self._lib.pa_alloc_admit(self._h, int(seq), int(n_tokens),
                                        -1 if share_src is None else int(share_src),
                                        int(n_shared)), "pa_alloc_admit")

    def ensure_capacity(self, seq: int, n_tokens: int) -> None:
        _check(self._lib.pa_alloc_ensure_capacity(self._h, int(seq), int(n_tokens)),
               "pa_alloc_ensure_capacity")

    def free_seq(self, seq: int) -> None:
        _check(self._lib.pa_alloc_free_seq(self._h, int(seq)), "pa_alloc_free_seq")

    def check_consistent(self) -> None:
        _check(self._lib.pa_alloc_check_consistent(self._h), "pa_alloc_check_consistent")

    @property
    def num_free(self) -> int:
        return int(self._lib.pa_alloc_num_free(self._h))

    def refcount(self, b: int) -> int:
        return int(self._lib.pa_alloc_refcount(self._h, int(b)))

    def table(self, seq: int) -> list:
        n = C.c_int32()
        _check(self._lib.pa_alloc_table(self._h, int(seq), None, 0, C.byref(n)), "pa_alloc_table")
        out = np.empty(max(n.value, 1), np.int32)
        _check(self._lib.pa_alloc_table(self._h, int(seq), _p32(out), n.value, C.byref(n)),
               "pa_alloc_table")
        return out[:n.value].tolist()

    def slots(self, seq: int, start: int, n: int) -> list:
        out = np.empty(max(n, 1), np.int32)
        _check(self._lib.pa_alloc_slots(self._h, int(seq), int(start), int(n), _p32(out)),
               "pa_alloc_slots")
        return out[:n].tolist()

    def trim(self, seq: int, n_tokens: int) -> None:
        _check(self._lib.pa_alloc_trim(self._h, int(seq), int(n_tokens)), "pa_alloc_trim")

    def fork(self, src: int, dst: int) -> None:
        _check(self._lib.pa_alloc_fork(self._h, int(src), int(dst)), "pa_alloc_fork")

    def cow(self, seq: int, start: int, n: int) -> list:
        """Private blocks for positions start..start+n-1; returns [(old, new)] block copies."""
        cap = max(n // self.block_size + 2, 1)
        pairs = np.empty(2 * cap, np.int32)
        k = C.c_int32()
        _check(self._lib.pa_alloc_cow(self._h, int(seq), int(start), int(n), _p32(pairs), cap,
                                      C.byref(k)), "pa_alloc_cow")
        return [(int(pairs[2 * i]), int(pairs[2 * i + 1])) for i in range(k.value)]

    def build_step(self, seqs, ctx_lens, n_new, max_blocks: int):
        """Returns (cu_seqlens_q, slot_mapping, block_table) host arrays for one step."""
        seqs, ctx_lens, n_new = _i32(seqs), _i32(ctx_lens), _i32(n_new)
        B = len(seqs)
        cu = np.zeros(B + 1, np.int32)
        T = int(n_new.sum())
        slots = np.empty(max(T, 1), np.int32)
        table = np.empty((max(B, 1), max_blocks), np.int32)
        _check(self._lib.pa_alloc_build_step(self._h, _p32(seqs), _p32(ctx_lens), _p32(n_new), B,
                                             _p32(cu), _p32(slots), _p32(table), int(max_blocks)),
               "pa_alloc_build_step")
        return cu, slots[:T], table[:B]


class Scheduler:
    """Owns a pa_scheduler: requests in, flat ragged steps out (see pagedattn.h)."""

    def __init__(self, num_blocks: int, block_size: int, chunk: int, budget: int):
        self._lib = load()
        h = C.c_void_p()
        _check(self._lib.pa_sched_create(int(num_blocks), int(block_size), int(chunk),
                                         int(budget), C.byref(h)), "pa_sched_create")
        self._h = h
        self._live = 0
        self.block_size = int(block_size)
        self.allocator = Allocator(num_blocks, block_size,
                                   _borrow=C.c_void_p(self._lib.pa_sched_allocator(h)))

    def close(self):
        if getattr(self, "_h", None):
            self.allocator._h = None
            self._lib.pa_sched_destroy(self._h)
            self._h = None

    __del__ = close

    def add(self, seq: int, prompt_len: int, max_new: int, leader: Optional[int] = None):
        _check(self._lib.pa_sched_add(self._h, int(seq), int(prompt_len), int(max_new),
                                      -1 if leader is None else int(leader)), "pa_sched_add")
        self._live += 1

    def step(self):
        """[(seq, n_new, ctx)] in step order."""
        cap = max(self._live, 1)
        seqs, n_new, ctx = (np.empty(cap, np.int32) for _ in range(3))
        n = C.c_int32()
        _check(self._lib.pa_sched_step(self._h, _p32(seqs), _p32(n_new), _p32(ctx), cap,
                                       C.byref(n)), "pa_sched_step")
        k = n.value
        return list(zip(seqs[:k].tolist(), n_new[:k].tolist(), ctx[:k].tolist()))

    def commit(self) -> list:
        cap = max(self._live, 1)
        fin = np.empty(cap, np.int32)
        n = C.c_int32()
        _check(self._lib.pa_sched_commit(self._h, _p32(fin), cap, C.byref(n)), "pa_sched_commit")
        self._live -= n.value
        return fin[:n.value].tolist()

    def counts(self):
        w, r, p = C.c_int32(), C.c_int32(), C.c_int64()
        _check(self._lib.pa_sched_counts(self._h, C.byref(w), C.byref(r), C.byref(p)),
               "pa_sched_counts")
        return int(w.value), int(r.value), int(p.value)

    def seq(self, q: int):
        """(n_tokens, num_computed, generated) of sequence q."""
        a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
        _check(self._lib.pa_sched_seq(self._h, int(q), C.byref(a), C.byref(b), C.byref(c)),
               "pa_sched_seq")
        return int(a.value), int(b.value), int(c.value)


# ------------------------------------------------------------------ host step metadata

def pa_compute_slots(shape: Shape, block_table: np.ndarray, cu_seqlens_q: np.ndarray,
                     ctx_lens: np.ndarray) -> np.ndarray:
    bt = _i32(block_table)
    cu, ctx = _i32(cu_seqlens_q), _i32(ctx_lens)
    B = len(ctx)
    T = int(cu[-1]) if B else 0
    out = np.empty(max(T, 1), np.int32)
    mb = bt.shape[1] if bt.ndim == 2 else 0
    _check(load().pa_compute_slots(C.byref(shape), _p32(bt), B, mb, _p32(cu), _p32(ctx),
                                   _p32(out)), "pa_compute_slots")
    return out[:T]


def pa_plan_step(shape: Shape, cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray) -> np.ndarray:
    """Work items for one step as a numpy structured array (dtype WORK_ITEM_DTYPE)."""
    lib = load()
    cu, ctx = _i32(cu_seqlens_q), _i32(ctx_lens)
    B = len(ctx)
    T = int(cu[-1]) if B else 0
    max_ctx = int(ctx.max()) if B else 0
    cap = int(lib.pa_plan_max_items(C.byref(shape), B, T, max_ctx))
    buf = (WorkItem * max(cap, 1))()
    n = C.c_int32()
    _check(lib.pa_plan_step(C.byref(shape), B, _p32(cu), _p32(ctx), buf, cap, C.byref(n)),
           "pa_plan_step")
    arr = np.frombuffer(buf, dtype=WORK_ITEM_DTYPE, count=max(cap, 1))[:n.value].copy()
    return arr


def pa_plan_step_shared(shape: Shape, cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray,
                        block_table: np.ndarray) -> np.ndarray:
    """Work items with prefix sharing (GROUP / RESUME items for decode rows whose tables share
    leading key tiles), as a numpy structured array (dtype WORK_ITEM_DTYPE)."""
    lib = load()
    cu, ctx, bt = _i32(cu_seqlens_q), _i32(ctx_lens), _i32(block_table)
    B = len(ctx)
    T = int(cu[-1]) if B else 0
    max_ctx = int(ctx.max()) if B else 0
    cap = int(lib.pa_plan_max_items_shared(C.byref(shape), B, T, max_ctx))
    buf = (WorkItem * max(cap, 1))()
    n = C.c_int32()
    mb = bt.shape[1] if bt.ndim == 2 else 0
    _check(lib.pa_plan_step_shared(C.byref(shape), B, _p32(cu), _p32(ctx), _p32(bt), mb, buf, cap,
                                   C.byref(n)), "pa_plan_step_shared")
    return np.frombuffer(buf, dtype=WORK_ITEM_DTYPE, count=max(cap, 1))[:n.value].copy()


def pa_workspace_bytes(shape: Shape, T: int, max_ctx: int) -> int:
    return int(load().pa_workspace_bytes(C.byref(shape), int(T), int(max_ctx)))


def pa_upload_block_table(shape: Shape, host: np.ndarray, dev, stream=None) -> None:
    h = _i32(host)
    B, mb = (h.shape if h.ndim == 2 else (0, 0))
    _check(load().pa_upload_block_table(C.byref(shape), _p32(h), _dev(dev), B, mb,
                                        _stream(stream)), "pa_upload_block_table")


# ------------------------------------------------------------------------- device step

def paged_copy_blocks(pairs, k_pool, v_pool, shape: Shape, err=None, stream=None) -> None:
    """pairs: device int32 tensor [2 * n] of (old, new) block ids from Allocator.cow."""
    n = int(pairs.numel() // 2)
    _check(load().paged_copy_blocks(_dev(pairs) if n else None, n, _dev(k_pool), _dev(v_pool),
                                    C.byref(shape), _dev(err), _stream(stream)),
           "paged_copy_blocks")


def paged_kv_write(k_new, v_new, slot_mapping, k_pool, v_pool, shape: Shape, err=None,
                   stream=None) -> None:
    T = int(slot_mapping.shape[0])
    _check(load().paged_kv_write(_dev(k_new), _dev(v_new), _dev(slot_mapping), T, _dev(k_pool),
                                 _dev(v_pool), C.byref(shape), _dev(err), _stream(stream)),
           "paged_kv_write")


def paged_attention_step(q, k_pool, v_pool, block_table, cu_seqlens_q, ctx_lens, max_ctx: int,
                         items, workspace, out, shape: Shape, err=None, stream=None) -> None:
    """items: a device int32 tensor holding the pa_work_item records from pa_plan_step."""
    B = int(ctx_lens.shape[0])
    T = int(q.shape[0])
    n_items = int(items.numel() // ITEM_INTS)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().paged_attention_step(
        _dev(q), _dev(k_pool), _dev(v_pool), _dev(block_table), int(block_table.shape[1]),
        _dev(cu_seqlens_q), _dev(ctx_lens), B, T, int(max_ctx), _dev(items), n_items,
        _dev(workspace), ws_bytes, _dev(out), C.byref(shape), _dev(err), _stream(stream)),
        "paged_attention_step")


def paged_kv_write_fp8(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale: float,
                       v_scale: float, shape: Shape, err=None, stream=None) -> None:
    """bf16 k_new / v_new [T, Hkv, D] quantised into uint8 float8_e4m3fn pools with per-tensor
    scales (code = e4m3(x / scale))."""
    T = int(slot_mapping.shape[0])
    _check(load().paged_kv_write_fp8(_dev(k_new), _dev(v_new), _dev(slot_mapping), T,
                                     _dev(k_pool), _dev(v_pool), float(k_scale), float(v_scale),
                                     C.byref(shape), _dev(err), _stream(stream)),
           "paged_kv_write_fp8")


def paged_attention_step_fp8(q, k_pool, v_pool, block_table, cu_seqlens_q, ctx_lens,
                             max_ctx: int, items, k_scale: float, v_scale: float, workspace,
                             out, shape: Shape, err=None, stream=None) -> None:
    """paged_attention_step over uint8 float8_e4m3fn pools with per-tensor scales."""
    B = int(ctx_lens.shape[0])
    T = int(q.shape[0])
    n_items = int(items.numel() // ITEM_INTS)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().paged_attention_step_fp8(
        _dev(q), _dev(k_pool), _dev(v_pool), _dev(block_table), int(block_table.shape[1]),
        _dev(cu_seqlens_q), _dev(ctx_lens), B, T, int(max_ctx), _dev(items), n_items,
        float(k_scale), float(v_scale), _dev(workspace), ws_bytes, _dev(out), C.byref(shape),
        _dev(err), _stream(stream)),
        "paged_attention_step_fp8")


class StepLimits:
    """Fixed sizes of a step that is captured in a CUDA graph: B sequences, T query rows,
    block-table width max_blocks and a context bound max_ctx. Every step prepared under these
    limits reuses the same device buffers and launches the same kernels with the same
    arguments, so a graph captured once replays any of them."""

    def __init__(self, B: int, T: int, max_blocks: int, max_ctx: int):
        self.B, self.T, self.max_blocks, self.max_ctx = int(B), int(T), int(max_blocks), int(max_ctx)


class StepRunner:
    """One layer's step on the device: holds the plan buffers and workspace, runs
    paged_kv_write then paged_attention_step on the current stream.

    prepare() takes host metadata (the plan is computed on the host); run() launches.
    With limits (StepLimits), prepare() writes the metadata into fixed device buffers in place
    (the plan padded to a fixed item count with n_q == 0 items, the table padded with -1), so
    capture() can record run() once in a CUDA graph and replay() runs any later prepared step.
    Those buffers are views of one device array, filled from one pinned host array by a single
    asynchronous copy on the current stream; the next prepare() first waits for that copy.
    With kv_scales = (k_scale, v_scale) the pools are uint8 float8_e4m3fn caches and the fp8
    write and read entry points run instead.
    """

    def __init__(self, shape: Shape, device="cuda", limits: Optional[StepLimits] = None,
                 kv_scales: Optional[tuple] = None):
        import torch
        self.torch = torch
        self.shape = shape
        self.kv_scales = None if kv_scales is None else (float(kv_scales[0]), float(kv_scales[1]))
        self.device = torch.device(device)
        self.limits = limits
        self.ws = None
        self.graph = None
        self.err = torch.zeros(1, dtype=torch.int32, device=self.device)
        if limits is not None:
            L = limits
            d = self.device
            cap = int(load().pa_plan_max_items_shared(C.byref(shape), L.B, L.T, L.max_ctx))
            self.n_items_cap = max(cap, 1)
            parts = (("items", self.n_items_cap * ITEM_INTS), ("cu", L.B + 1), ("ctx", L.B),
                     ("table", L.B * L.max_blocks), ("slots", L.T))
            total = sum(n for _, n in parts)
            self._meta = torch.empty(max(total, 1), dtype=torch.int32, device=d)
            on_gpu = self.device.type == "cuda"
            self._h_meta = torch.empty(max(total, 1), dtype=torch.int32, pin_memory=on_gpu)
            h = self._h_meta.numpy()
            self._h, dev, off = {}, {}, 0
            for name, n in parts:
                self._h[name], dev[name] = h[off:off + n], self._meta[off:off + n]
                off += n
            self._h["table"] = self._h["table"].reshape(L.B, L.max_blocks)
            h[:] = 0                                      # items: n_q == 0, padding
            self._h["table"].fill(-1)
            self._h["slots"].fill(-1)
            self._meta.copy_(self._h_meta)
            self.items, self.cu, self.ctx = dev["items"], dev["cu"], dev["ctx"]
            self.table = dev["table"].view(L.B, L.max_blocks)
            self.slots = dev["slots"]
            self._uploaded = None                         # event after the last upload
            self._n_planned = 0                           # real items of the last plan
            self.max_ctx = L.max_ctx
            self.T = L.T
            need = pa_workspace_bytes(shape, L.T, L.max_ctx)
            self.ws = torch.empty((need + 3) // 4, dtype=torch.float32, device=d)

    def prepare(self, cu_seqlens_q: np.ndarray, ctx_lens: np.ndarray, block_table: np.ndarray,
                slot_mapping: Optional[np.ndarray] = None):
        torch = self.torch
        cu, ctx = _i32(cu_seqlens_q), _i32(ctx_lens)
        if self.limits is not None:
            return self._prepare_fixed(cu, ctx, _i32(block_table), slot_mapping)
        items = pa_plan_step_shared(self.shape, cu, ctx, block_table)
        if slot_mapping is None:
            slot_mapping = pa_compute_slots(self.shape, block_table, cu, ctx)
        d = self.device
        self.max_ctx = int(ctx.max()) if len(ctx) else 0
        self.T = int(cu[-1]) if len(ctx) else 0
        self.items = torch.from_numpy(items.view(np.int32).reshape(-1).copy()).to(d)
        self.cu = torch.from_numpy(cu.copy()).to(d)
        self.ctx = torch.from_numpy(ctx.copy()).to(d)
        self.table = torch.from_numpy(_i32(block_table).copy()).to(d)
        self.slots = torch.from_numpy(_i32(slot_mapping).copy()).to(d)
        need = pa_workspace_bytes(self.shape, self.T, self.max_ctx)
        if self.ws is None or self.ws.numel() * 4 < need:
            self.ws = torch.empty((need + 3) // 4, dtype=torch.float32, device=d)
        return self

    def _prepare_fixed(self, cu, ctx, table, slot_mapping):
        """prepare() under limits: the plan and the slots are written by the library straight into
        the pinned host array, which then goes to the device in one copy."""
        L = self.limits
        B = len(ctx)
        T = int(cu[-1]) if B else 0
        if B != L.B or T != L.T or table.ndim != 2 or table.shape[0] != B or \
                table.shape[1] > L.max_blocks or (B and int(ctx.max()) > L.max_ctx):
            raise ValueError("step exceeds the limits the runner was built for")
        if self._uploaded is not None:
            self._uploaded.synchronize()                  # the pinned array is free again
        lib = load()
        hi = self._h["items"]
        n = C.c_int32()
        _check(lib.pa_plan_step_shared(C.byref(self.shape), B, _p32(cu), _p32(ctx), _p32(table),
                                       table.shape[1], hi.ctypes.data_as(C.POINTER(WorkItem)),
                                       self.n_items_cap, C.byref(n)), "pa_plan_step_shared")
        hs = hi.view(WORK_ITEM_DTYPE)
        if self._n_planned > n.value:
            hs[n.value:self._n_planned] = 0               # n_q == 0: padding
        self._n_planned = n.value
        self._h["cu"][:] = cu
        self._h["ctx"][:] = ctx
        ht = self._h["table"]
        ht[:, :table.shape[1]] = table
        if table.shape[1] < L.max_blocks:
            ht[:, table.shape[1]:] = -1
        if slot_mapping is not None:
            self._h["slots"][:] = _i32(slot_mapping)
        elif T > 0:
            _check(lib.pa_compute_slots(C.byref(self.shape), _p32(table), B, table.shape[1],
                                        _p32(cu), _p32(ctx), _p32(self._h["slots"])),
                   "pa_compute_slots")
        self._meta.copy_(self._h_meta, non_blocking=True)
        if self._meta.is_cuda:
            self._uploaded = self.torch.cuda.Event()
            self._uploaded.record()
        return self

    @property
    def meta_bytes(self) -> int:
        """Bytes prepare() copies to the device per step (limits mode: the whole padded array)."""
        if self.limits is not None:
            return int(self._meta.numel()) * 4
        return 4 * int(self.items.numel() + self.cu.numel() + self.ctx.numel() +
                       self.table.numel() + self.slots.numel())

    def capture(self, q, k_new, v_new, k_pool, v_pool, out, write: bool = True,
                attend: bool = True):
        """Records run() (or only its write or attention part) in a CUDA graph. Needs limits;
        the tensors passed here are the ones every replay reads and writes."""
        torch = self.torch
        if self.limits is None:
            raise ValueError("capture needs a runner built with StepLimits")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):              # warm-up outside the graph
            if write:
                self.write(k_new, v_new, k_pool, v_pool)
            if attend:
                self.attend(q, k_pool, v_pool, out)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            if write:
                self.write(k_new, v_new, k_pool, v_pool)
            if attend:
                self.attend(q, k_pool, v_pool, out)
        self.graph = graph
        return graph

    def replay(self):
        self.graph.replay()

    def write(self, k_new, v_new, k_pool, v_pool, stream=None):
        if self.kv_scales is not None:
            paged_kv_write_fp8(k_new, v_new, self.slots, k_pool, v_pool, *self.kv_scales,
                               self.shape, self.err, stream)
            return
        paged_kv_write(k_new, v_new, self.slots, k_pool, v_pool, self.shape, self.err, stream)

    def attend(self, q, k_pool, v_pool, out, stream=None):
        if self.kv_scales is not None:
            paged_attention_step_fp8(q, k_pool, v_pool, self.table, self.cu, self.ctx,
                                     self.max_ctx, self.items, *self.kv_scales, self.ws, out,
                                     self.shape, self.err, stream)
            return
        paged_attention_step(q, k_pool, v_pool, self.table, self.cu, self.ctx, self.max_ctx,
                             self.items, self.ws, out, self.shape, self.err, stream)

    def run(self, q, k_new, v_new, k_pool, v_pool, out, stream=None):
        self.write(k_new, v_new, k_pool, v_pool, stream)
        self.attend(q, k_pool, v_pool, out, stream)
        return out

    def device_error(self) -> int:
        return int(self.err.item())


class StepPipeline:
    """A stream of steps under fixed limits, run end to end from host buffers by the library's
    native pipeline (pa_pipeline_* in pagedattn.h): per step one call plans the step into
    pinned metadata and queues the uploads, the captured KV write + attention and the read of
    the output, so that one step's host work and copies overlap the kernels of the step before
    it. k_pool / v_pool are the device pools every step writes and reads (bf16, or uint8 codes
    with kv_scales)."""

    class Pending:
        """A submitted step; synchronize() returns once its output is in its host buffer."""

        def __init__(self, pipe, slot):
            self.pipe, self.slot = pipe, slot

        def synchronize(self):
            _check(self.pipe._lib.pa_pipeline_wait(self.pipe._h, self.slot), "pa_pipeline_wait")

    def __init__(self, shape: Shape, limits: StepLimits, k_pool, v_pool,
                 kv_scales: Optional[tuple] = None):
        self._lib = load()
        self.shape, self.limits = shape, limits
        self._pools = (k_pool, v_pool)                # kept alive as long as the pipeline
        L = limits
        fp8 = kv_scales is not None
        ks, vs = (float(kv_scales[0]), float(kv_scales[1])) if fp8 else (1.0, 1.0)
        h = C.c_void_p()
        _check(self._lib.pa_pipeline_create(C.byref(shape), L.B, L.T, L.max_blocks, L.max_ctx,
                                            _dev(k_pool), _dev(v_pool), 1 if fp8 else 0, ks, vs,
                                            C.byref(h)), "pa_pipeline_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_pipeline_destroy(self._h)
            self._h = None

    __del__ = close

    @property
    def meta_bytes(self) -> int:
        return int(self._lib.pa_pipeline_meta_bytes(self._h))

    def submit(self, cu_seqlens_q, ctx_lens, block_table, h_q, h_k_new, h_v_new, h_out):
        """Queues one step; h_* are host tensors (pinned for asynchronous copies): q and out
        [T, Hq, D], k_new and v_new [T, Hkv, D], bf16 (or int16 bit patterns). Returns a
        Pending whose synchronize() returns once h_out holds the step's output."""
        cu, ctx, table = _i32(cu_seqlens_q), _i32(ctx_lens), _i32(block_table)
        slot = C.c_int32()
        _check(self._lib.pa_pipeline_submit(self._h, _p32(cu), _p32(ctx), _p32(table),
                                            int(table.shape[1]), h_q.data_ptr(),
                                            h_k_new.data_ptr(), h_v_new.data_ptr(),
                                            h_out.data_ptr(), C.byref(slot)),
               "pa_pipeline_submit")
        return StepPipeline.Pending(self, int(slot.value))

    def device_error(self) -> int:
        e = C.c_int32()
        _check(self._lib.pa_pipeline_device_error(self._h, C.byref(e)), "pa_pipeline_device_error")
        return int(e.value)
