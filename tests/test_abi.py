"""The C-ABI library on the CPU: it loads, exports every symbol include/pagedattn.h declares,
and its host-side step metadata is bit-exact against the oracle (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from continuous_batching_gb300 import build
    build.build()                     # incremental: recompiles only what changed
    return bd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?(?:int32_t|int64_t|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(",
                      text, flags=re.M)


def test_every_declared_symbol_is_exported(built_library):
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(bd.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version_and_status_strings():
    assert bd.pa_abi_version() == 3
    assert bd.status_string(bd.PA_ERR_OOM) == "PA_ERR_OOM"
    assert bd.status_string(999) == "PA_ERR_UNKNOWN"


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_slot_mapping_matches_oracle(name):
    st = wl.make_config(name, with_pool=False)
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    got = bd.pa_compute_slots(shape, st.block_table, st.cu_seqlens_q, st.ctx_lens)
    want = pa.slot_mapping(st.block_table, st.cu_seqlens_q, st.ctx_lens, st.block_size)
    assert got.dtype == np.int32 and np.array_equal(got.astype(np.int64), want)


def test_slot_mapping_rejects_bad_metadata():
    st = wl.make_config("tiny", with_pool=False)
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    bad = st.block_table.copy()
    bad[0, 0] = st.num_blocks                    # outside the pool
    with pytest.raises(bd.PagedAttnError):
        bd.pa_compute_slots(shape, bad, st.cu_seqlens_q, st.ctx_lens)
    cu = st.cu_seqlens_q.copy()
    cu[2] = cu[1] - 1                            # decreasing
    with pytest.raises(bd.PagedAttnError):
        bd.pa_compute_slots(shape, st.block_table, cu, st.ctx_lens)
    ctx = st.ctx_lens.copy()
    ctx[0] = 0                                   # fewer keys than query rows
    with pytest.raises(bd.PagedAttnError):
        bd.pa_compute_slots(shape, st.block_table, st.cu_seqlens_q, ctx)
    with pytest.raises(bd.PagedAttnError):       # unsupported head_dim
        bd.pa_compute_slots(bd.Shape.make(4, 2, 96, 16, 32), st.block_table, st.cu_seqlens_q,
                            st.ctx_lens)


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_plan_covers_every_row_head_split_once(name):
    """Each (query row, KV head, split s <= pos // PA_SPLIT_TOKENS) appears in exactly one item. A decode
    row's splits are items of one split each; a prefill tile's item starts at split 0 and
    covers every split its last row reaches."""
    st = wl.make_config(name, with_pool=False)
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    items = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)
    g = st.Hq // st.Hkv
    seq_of, pos_of = pa.row_positions(st.cu_seqlens_q, st.ctx_lens)
    nsplit = pos_of // bd.PA_SPLIT_TOKENS + 1
    count = {}
    for it in items:
        assert 1 <= it["n_q"] <= 128 // g
        cu0, cu1 = st.cu_seqlens_q[it["seq"]], st.cu_seqlens_q[it["seq"] + 1]
        assert cu0 <= it["q_start"] and it["q_start"] + it["n_q"] <= cu1
        last = it["q_start"] + it["n_q"] - 1
        if cu1 - cu0 == 1:
            assert it["n_splits"] == 1
        else:
            assert it["split"] == 0 and it["n_splits"] == nsplit[last]
        # tiles of 128 keys from the item's first split up to its last row's position
        k0 = it["split"] * bd.PA_SPLIT_TOKENS
        k1 = min(k0 + it["n_splits"] * bd.PA_SPLIT_TOKENS, pos_of[last] + 1)
        assert it["n_tiles"] == -(-(k1 - k0) // bd.PA_TILE_KEYS)
        for t in range(it["q_start"], it["q_start"] + it["n_q"]):
            for sp in range(it["split"], it["split"] + it["n_splits"]):
                if sp < nsplit[t]:
                    key = (t, it["kv_head"], sp)
                    count[key] = count.get(key, 0) + 1
    want = {(t, h, s) for t in range(st.T) for h in range(st.Hkv) for s in range(nsplit[t])}
    assert set(count) == want and all(v == 1 for v in count.values())
    check_lists(items, len(items))
    again = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)     # deterministic
    assert np.array_equal(items, again)


def walk(items, n_items):
    """The kernel's walk: CTA c of min(n_items, PA_PLAN_CTAS) starts at item c and follows
    `next` (<= 0 ends) while it moves forward; padding (n_q == 0) ends a list."""
    lists = []
    for c in range(min(n_items, bd.PA_PLAN_CTAS)):
        got, idx = [], c
        while 0 <= idx < n_items and items[idx]["n_q"] != 0:
            got.append(idx)
            nxt = int(items[idx]["next"])
            assert nxt <= 0 or idx < nxt < n_items, "a link must move forward"
            idx = nxt if nxt > 0 else -1
        lists.append(got)
    return lists


def check_lists(items, n_items):
    """Every real item is on exactly one list; the layout and the longest-processing-time
    deal the planner documents."""
    n = int(np.sum(items["n_q"][:n_items] != 0))
    G = min(n, bd.PA_PLAN_CTAS)
    lists = walk(items, n_items)
    seen = [i for L in lists for i in L]
    assert sorted(seen) == list(range(n)), "each real item once, padding never"
    assert all(len(L) > 0 for L in lists[:G]) and all(not L for L in lists[G:])
    # stored position by position: the k-th items of all lists, lists in order
    order = [L[k] for k in range(max(map(len, lists), default=0)) for L in lists if k < len(L)]
    assert order == list(range(n))
    tiles = items["n_tiles"][:n].astype(np.int64)
    cost = [int(np.sum(tiles[L] + 1)) for L in lists[:G]]
    for L in lists[:G]:
        assert np.all(np.diff(tiles[L]) <= 0), "a list takes its items longest first"
    if G:
        # the greedy deal: when a list took its last item it was the cheapest list, so it
        # exceeds the cheapest final list by at most that item's cost
        for L, c in zip(lists[:G], cost):
            assert c - (tiles[L[-1]] + 1) <= min(cost)
        # the longest G items open the G lists, longest first
        assert np.all(np.diff(tiles[:G]) <= 0)
        assert tiles[:G].min() >= (tiles[G:].max() if n > G else 0)


def test_plan_lists_balance_a_skewed_step():
    """One long prefill segment among many short decodes: the deal puts the long items on
    lists of their own and keeps the busiest list near the average."""
    ctx = [9000 + 512] + [300] * 400
    nq = [512] + [1] * 400
    cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    shape = bd.Shape.make(32, 8, 128, 16, 4096)
    items = bd.pa_plan_step(shape, cu, np.array(ctx, np.int32))
    check_lists(items, len(items))
    lists = walk(items, len(items))
    cost = [int(np.sum(items["n_tiles"][L].astype(np.int64) + 1)) for L in lists]
    longest = int(items["n_tiles"].max()) + 1
    assert max(cost) <= max(np.mean(cost), longest) + longest


def test_padded_plan_walk_covers_the_real_items_once():
    """A plan padded to a fixed count (a captured step): the CTAs past the real plan's lists
    start at padding and do nothing."""
    shape = bd.Shape.make(32, 8, 128, 16, 4096)
    for ctx, nq in (([40, 3000], [1, 1]), ([5000] * 30, [1] * 30), ([700, 900], [300, 1])):
        cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
        items = bd.pa_plan_step(shape, cu, np.array(ctx, np.int32))
        cap = int(bd.load().pa_plan_max_items(ctypes.byref(shape), len(ctx), int(cu[-1]),
                                              max(ctx)))
        assert cap >= len(items)
        padded = np.zeros(cap, dtype=bd.WORK_ITEM_DTYPE)
        padded[:len(items)] = items
        check_lists(padded, cap)


def test_header_constants_match_the_binding():
    import os, re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "pagedattn.h")).read()
    defs = dict(re.findall(r"#define (PA_\w+)\s+(\d+)", hdr))
    for name in ("PA_SPLIT_TOKENS", "PA_TILE_KEYS", "PA_PLAN_CTAS", "PA_DEVERR_BLOCK",
                 "PA_DEVERR_SLOT", "PA_DEVERR_TIMEOUT", "PA_DEVERR_META"):
        assert int(defs[name]) == getattr(bd, name), name


def test_workspace_bytes_cover_partials():
    shape = bd.Shape.make(32, 8, 128, 16, 100)
    assert bd.pa_workspace_bytes(shape, 10, 3000) == 10 * 2 * 32 * 130 * 4
    assert bd.pa_workspace_bytes(shape, 10, 4097) == 10 * 3 * 32 * 130 * 4
    assert bd.pa_workspace_bytes(shape, 0, 0) == 256


def test_upload_rejects_out_of_range_table_without_gpu():
    """Validation happens on the host before any copy, so it needs no device."""
    shape = bd.Shape.make(4, 2, 64, 16, 8)
    bad = np.array([[0, 9]], np.int32)
    st = bd.load().pa_upload_block_table(ctypes.byref(shape), bad.ctypes.data_as(bd._i32p),
                                         None, 1, 2, None)
    assert st == bd.PA_ERR_BOUNDS


def test_limits_runner_lays_out_padded_metadata_without_gpu():
    """StepRunner with StepLimits: one metadata array whose views hold the plan padded with
    n_q == 0 items, cu / ctx, the table padded with -1 and the slots; a second, smaller step
    prepared into the same buffers leaves no stale entries. (Host logic: a CPU 'device'.)"""
    torch = pytest.importorskip("torch")
    shape = bd.Shape.make(8, 2, 64, 16, 64)
    lim = bd.StepLimits(B=3, T=5, max_blocks=6, max_ctx=90)
    r = bd.StepRunner(shape, device="cpu", limits=lim)
    steps = [([40, 90, 17], [1, 3, 1],
              [[0, 1, 2, -1, -1, -1], [3, 4, 5, 6, 7, 8], [9, 10, -1, -1, -1, -1]]),
             ([16, 20, 33], [2, 2, 1], [[11, -1, -1], [12, 13, -1], [14, 15, 16]])]
    for ctx, nq, tab in steps:
        ctx = np.array(ctx, np.int32)
        cu = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
        tab = np.array(tab, np.int32)
        r.prepare(cu, ctx, tab)
        items = bd.pa_plan_step(shape, cu, ctx)
        dev_items = r.items.numpy().view(bd.WORK_ITEM_DTYPE)
        assert len(dev_items) == r.n_items_cap >= len(items)
        assert np.array_equal(dev_items[:len(items)], items)
        assert np.all(dev_items["n_q"][len(items):] == 0) and np.all(dev_items[len(items):]["next"] == 0)
        assert np.array_equal(r.cu.numpy(), cu) and np.array_equal(r.ctx.numpy(), ctx)
        want = np.full((3, 6), -1, np.int32)
        want[:, :tab.shape[1]] = tab
        assert np.array_equal(r.table.numpy(), want)
        assert np.array_equal(r.slots.numpy(), bd.pa_compute_slots(shape, tab, cu, ctx))
        assert r.meta_bytes == 4 * (r.n_items_cap * bd.ITEM_INTS + 4 + 3 + 18 + 5)
    with pytest.raises(ValueError):
        r.prepare(np.array([0, 1, 2], np.int32), np.array([5, 5], np.int32), np.zeros((2, 1), np.int32))


def test_limits_runner_clears_items_of_a_longer_previous_plan_without_gpu():
    """A plan with fewer items than the one before it: the items past its end read as padding
    again (the kernel's CTAs past the plan's lists start there)."""
    pytest.importorskip("torch")
    shape = bd.Shape.make(8, 2, 64, 16, 1024)
    lim = bd.StepLimits(B=2, T=2, max_blocks=320, max_ctx=5000)
    r = bd.StepRunner(shape, device="cpu", limits=lim)
    cu = np.array([0, 1, 2], np.int32)
    table = np.arange(640, dtype=np.int32).reshape(2, 320)
    counts = []
    for ctx in ([4500, 5000], [100, 200], [5000, 17]):
        ctx = np.array(ctx, np.int32)
        r.prepare(cu, ctx, table)
        items = bd.pa_plan_step(shape, cu, ctx)
        dev = r.items.numpy().view(bd.WORK_ITEM_DTYPE)
        assert np.array_equal(dev[:len(items)], items)
        assert not np.any(dev.view(np.int32).reshape(len(dev), bd.ITEM_INTS)[len(items):])
        assert np.array_equal(r.slots.numpy(), bd.pa_compute_slots(shape, table, cu, ctx))
        check_lists(dev, len(dev))
        counts.append(len(items))
    assert counts[0] > counts[1] < counts[2]


# ------------------------------------------------------------ prefix sharing in the plan

def _tiles_covered(items, st):
    """(token, kv head) -> list of key tiles the items give it (GROUP items: tiles [0, tile0)
    of split 0 for each member row; RESUME: [tile0, end of split 0); PLAIN: its splits)."""
    seq_of, pos_of = pa.row_positions(st.cu_seqlens_q, st.ctx_lens)
    cov = {}
    T_SPLIT = bd.PA_SPLIT_TOKENS // bd.PA_TILE_KEYS
    for it in items:
        rows = range(it["q_start"], it["q_start"] + it["n_q"])
        for t in rows:
            last_tile = int(pos_of[t]) // bd.PA_TILE_KEYS
            if it["kind"] == bd.PA_ITEM_GROUP:
                tiles = range(0, int(it["tile0"]))
            elif it["kind"] == bd.PA_ITEM_RESUME:
                tiles = range(int(it["tile0"]), min(T_SPLIT - 1, last_tile) + 1)
            else:
                lo = int(it["split"]) * T_SPLIT
                hi = (int(it["split"]) + max(int(it["n_splits"]), 1)) * T_SPLIT
                tiles = range(lo, min(hi - 1, last_tile) + 1)
            cov.setdefault((t, int(it["kv_head"])), []).extend(tiles)
    return cov, pos_of


@pytest.mark.parametrize("name", wl.CONFIG_NAMES)
def test_shared_plan_covers_every_key_tile_once(name):
    st = wl.make_config(name, with_pool=False)
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    items = bd.pa_plan_step_shared(shape, st.cu_seqlens_q, st.ctx_lens, st.block_table)
    cov, pos_of = _tiles_covered(items, st)
    for t in range(st.T):
        for h in range(st.Hkv):
            want = list(range(int(pos_of[t]) // bd.PA_TILE_KEYS + 1))
            assert sorted(cov[(t, h)]) == want, (t, h)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    if name == "prefix":
        # 16 prompts x 8 samples sharing 64 blocks of 16 tokens: one group of 8 rows per
        # prompt and KV head over the 8 shared tiles
        assert len(groups) == 16 * st.Hkv
        assert np.all(groups["n_q"] == 8) and np.all(groups["tile0"] == 8)
        assert np.sum(items["kind"] == bd.PA_ITEM_RESUME) == 128 * st.Hkv
    else:
        # no block is shared: the plan is pa_plan_step's
        assert len(groups) == 0
        assert np.array_equal(items, bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens))
    # every real item on exactly one list; a group's RESUME items follow it on its list
    lists = walk(items, len(items))
    real = np.flatnonzero(items["n_q"] != 0).tolist()
    assert sorted(i for L in lists for i in L) == real
    where = {i: (c, k) for c, L in enumerate(lists) for k, i in enumerate(L)}
    for gi in np.flatnonzero(items["kind"] == bd.PA_ITEM_GROUP):
        g_it = items[gi]
        c, k = where[int(gi)]
        members = range(int(g_it["seq"]), int(g_it["seq"]) + int(g_it["n_q"]))
        nxt = lists[c][k + 1:k + 1 + len(members)]
        assert [int(items[j]["seq"]) for j in nxt] == list(members)
        assert all(items[j]["kind"] == bd.PA_ITEM_RESUME and items[j]["kv_head"] == g_it["kv_head"]
                   and items[j]["tile0"] == g_it["tile0"] for j in nxt)


def test_shared_plan_needs_two_whole_shared_tiles():
    """Decode rows whose tables agree on one 128-key tile only, or on blocks that do not fill a
    tile, stay PLAIN; rows that agree on two tiles form a group whose tile0 is the tiles all
    of them share."""
    shape = bd.Shape.make(32, 8, 128, 16, 4096)
    ctx = np.array([900, 900, 900], np.int32)
    cu = np.arange(4, dtype=np.int32)
    table = np.arange(3 * 64, dtype=np.int32).reshape(3, 64)
    table[1, :8] = table[0, :8]                                   # one tile in common
    items = bd.pa_plan_step_shared(shape, cu, ctx, table)
    assert np.all(items["kind"] == bd.PA_ITEM_PLAIN)
    table[1, :20] = table[0, :20]                                 # 2.5 tiles in common
    table[2, :40] = table[0, :40]                                 # 5 tiles
    items = bd.pa_plan_step_shared(shape, cu, ctx, table)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    assert len(groups) == 8 and np.all(groups["n_q"] == 3) and np.all(groups["tile0"] == 2)
    # 8 lists (one group per KV head) for 32 items: CTAs 8 .. 151 start at padding
    lists = walk(items, len(items))
    assert len(items) == 32 + bd.PA_PLAN_CTAS - 8
    assert all(L for L in lists[:8]) and not any(lists[8:])
    assert sorted(i for L in lists for i in L) == np.flatnonzero(items["n_q"] != 0).tolist()


def _check_shared_plan(shape, cu, ctx, table):
    """Plans with sharing, checks that every (row, KV head) gets each of its key tiles exactly
    once and that the plan's lists hold every real item once; returns the items."""
    from types import SimpleNamespace
    items = bd.pa_plan_step_shared(shape, cu, ctx, table)
    st = SimpleNamespace(cu_seqlens_q=cu, ctx_lens=ctx, T=int(cu[-1]), Hkv=shape.num_kv_heads)
    cov, pos_of = _tiles_covered(items, st)
    for t in range(st.T):
        for h in range(st.Hkv):
            assert sorted(cov[(t, h)]) == list(range(int(pos_of[t]) // bd.PA_TILE_KEYS + 1))
    lists = walk(items, len(items))
    assert sorted(i for L in lists for i in L) == np.flatnonzero(items["n_q"] != 0).tolist()
    return items


def test_shared_plan_groups_stop_at_the_row_limit_and_at_other_rows():
    """At g = 16 a tile holds 8 decode rows: 20 sequences sharing a prompt form groups of 8, 8
    and 4. A prefill row between samples of one prompt ends the run, and a later run of the
    same prompt forms a group of its own."""
    shape = bd.Shape.make(16, 1, 128, 16, 1 << 14)
    rng = np.random.default_rng(7)
    B = 20
    ctx = (512 + rng.integers(1, 700, size=B)).astype(np.int32)
    cu = np.arange(B + 1, dtype=np.int32)
    table = (np.arange(B * 96, dtype=np.int32).reshape(B, 96) + 64)
    table[:, :32] = np.arange(32)                                 # 512 tokens = 4 tiles shared
    items = _check_shared_plan(shape, cu, ctx, table)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    assert sorted(groups["n_q"].tolist()) == [4, 8, 8] and np.all(groups["tile0"] == 4)
    # sequence 5 becomes a 10-row prefill chunk between the samples
    n_q = np.ones(B, np.int32)
    n_q[5] = 10
    cu2 = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
    items = _check_shared_plan(shape, cu2, ctx, table)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    assert sorted((int(g["seq"]), int(g["n_q"])) for g in groups) == [(0, 5), (6, 8), (14, 6)]
    assert not np.any((items["kind"] != bd.PA_ITEM_PLAIN) & (items["seq"] == 5))


def test_shared_plan_tiles_stop_at_split_0_and_at_every_members_last_key():
    """A 4096-token shared prompt: the group takes the first 15 tiles (split 0 keeps one for
    each RESUME item), later splits are PLAIN items. A sample whose context ends 600 tokens in
    limits the group to the 4 whole tiles below its last key."""
    shape = bd.Shape.make(32, 8, 128, 16, 1 << 14)
    ctx = np.array([5000, 4500, 4200], np.int32)
    cu = np.arange(4, dtype=np.int32)
    table = np.arange(3 * 320, dtype=np.int32).reshape(3, 320) + 256
    table[:, :256] = np.arange(256)                              # 4096 tokens shared
    items = _check_shared_plan(shape, cu, ctx, table)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    assert len(groups) == 8 and np.all(groups["tile0"] == 15) and np.all(groups["n_q"] == 3)
    res = items[items["kind"] == bd.PA_ITEM_RESUME]
    assert len(res) == 24 and np.all(res["n_tiles"] == 1)
    ctx[1] = 600
    items = _check_shared_plan(shape, cu, ctx, table)
    groups = items[items["kind"] == bd.PA_ITEM_GROUP]
    assert len(groups) == 8 and np.all(groups["tile0"] == 4)
