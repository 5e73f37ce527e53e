"""GPU parity of the hot path through the C ABI: KV write bit-exact against the oracle, bf16
attention within max|diff| <= 1.5e-2 and mean|diff| <= 2e-3 of the fp64 oracle, on small
cases in full and on the five named workloads at full size (sampled rows)."""
import ctypes as C

import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, pool_np, run_step, shape_of

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def oracle_full(st):
    return pa.step(st.q, st.k_new, st.v_new, st.k_pool, st.v_pool, st.block_table,
                   st.cu_seqlens_q, st.ctx_lens, st.Hq, st.block_size)


def test_tiny_config_all_rows():
    st = wl.make_config("tiny")
    out, kp, vp, err = run_step(st, torch)
    slots, kp_ref, vp_ref, ref = oracle_full(st)
    assert err == 0
    assert np.array_equal(pool_np(kp, torch), kp_ref)
    assert np.array_equal(pool_np(vp, torch), vp_ref)
    assert_close(out, ref, "tiny")


# ragged mix: decode rows at tile and split boundaries plus prefill segments that start at 0,
# straddle the first split boundary, end on a tile boundary and have ragged tails
MID_CTX = [1, 17, 127, 128, 129, 1023, 1024, 1025, 2047, 2048, 2049, 4097, 200, 2100, 4200, 5, 384]
MID_NQ = [1] * 12 + [200, 77, 33, 5, 129]


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(32, 8, 128, 16), (8, 8, 128, 32), (16, 2, 64, 8),
                                         (64, 8, 128, 64), (16, 1, 128, 128), (4, 2, 64, 16),
                                         (32, 8, 128, 8), (64, 4, 128, 16), (32, 2, 64, 128)])
def test_mixed_step_all_rows(Hq, Hkv, D, bs):
    st = wl.make_step(Hq, Hkv, D, bs, MID_CTX, MID_NQ, seed=Hq * 7 + D + bs)
    out, kp, vp, err = run_step(st, torch)
    slots, kp_ref, vp_ref, ref = oracle_full(st)
    assert err == 0
    assert np.array_equal(pool_np(kp, torch), kp_ref)
    assert np.array_equal(pool_np(vp, torch), vp_ref)
    assert_close(out, ref, f"mixed Hq{Hq} Hkv{Hkv} D{D} bs{bs}")


def _sample_rows(st, rng, n=24):
    rows = set()
    for s in range(st.B):
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        if b - a > 1:
            rows.update([a, b - 1, a + (b - a) // 2])
    rows.update(rng.choice(st.T, size=min(n, st.T), replace=False).tolist())
    long_s = int(np.argmax(st.ctx_lens))
    rows.add(int(st.cu_seqlens_q[long_s + 1]) - 1)
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["decode", "mixed", "longtail", "prefix"])
def test_full_size_workloads_sampled(name):
    st = wl.make_config(name)
    out, kp, vp, err = run_step(st, torch)
    assert err == 0
    slots = pa.slot_mapping(st.block_table, st.cu_seqlens_q, st.ctx_lens, st.block_size)
    kp_np, vp_np = pool_np(kp, torch), pool_np(vp, torch)
    # the written slots carry the new rows bit-exactly; a sample of other blocks is untouched
    flat_k = kp_np.reshape(-1, st.Hkv, st.D)
    flat_v = vp_np.reshape(-1, st.Hkv, st.D)
    assert np.array_equal(flat_k[slots], st.k_new) and np.array_equal(flat_v[slots], st.v_new)
    rng = np.random.default_rng(1234)
    untouched = np.setdiff1d(np.arange(flat_k.shape[0]), slots)
    pick = rng.choice(untouched, size=min(4096, len(untouched)), replace=False)
    assert np.array_equal(flat_k[pick], st.k_pool.reshape(-1, st.Hkv, st.D)[pick])
    rows = _sample_rows(st, rng)
    ref = pa.attention_rows(st.q, kp_np, vp_np, st.block_table, st.cu_seqlens_q, st.ctx_lens,
                            st.Hq, rows)
    assert_close(out[rows], ref, name)
    assert np.all(np.isfinite(pa.bf16_to_f64(out)))


def test_longest_context_and_late_prefill_chunk():
    """ctx 40960 decode row and a 512-row chunk at prior offset 40448 (40 splits)."""
    st = wl.make_step(64, 8, 128, 32, [40960, 40960], [1, 512], seed=77)
    out, kp, vp, err = run_step(st, torch)
    assert err == 0
    rows = np.array([0, 1, 2, 100, 256, 511, 512])
    ref = pa.attention_rows(st.q, pool_np(kp, torch), pool_np(vp, torch), st.block_table,
                            st.cu_seqlens_q, st.ctx_lens, st.Hq, rows)
    assert_close(out[rows], ref, "ctx 40960")


def test_empty_step_and_zero_row_sequences():
    st = wl.make_step(8, 2, 128, 16, [40, 10, 300], [0, 0, 0], seed=3)
    out, kp, vp, err = run_step(st, torch)
    assert out.shape[0] == 0 and err == 0
    st = wl.make_step(8, 2, 128, 16, [40, 10, 300, 7], [0, 3, 0, 1], seed=4)
    out, kp, vp, err = run_step(st, torch)
    slots, kp_ref, vp_ref, ref = oracle_full(st)
    assert_close(out, ref, "zero-row sequences")


def test_stale_nan_in_pool_is_never_read():
    """Slots past each sequence's context hold NaN bit patterns: outputs stay finite and
    bit-identical to a pool holding ordinary stale values."""
    st = wl.make_step(32, 8, 128, 16, [5, 130, 1030, 17], [1, 1, 3, 17], seed=9)
    clean, _, _, _ = run_step(st, torch)
    kp = st.k_pool.copy()
    vp = st.v_pool.copy()
    flat_k = kp.reshape(-1, st.Hkv, st.D)
    flat_v = vp.reshape(-1, st.Hkv, st.D)
    live = set()
    for s in range(st.B):
        for p in range(int(st.ctx_lens[s])):
            live.add(int(st.block_table[s, p // st.block_size]) * st.block_size + p % st.block_size)
    dead = np.array(sorted(set(range(flat_k.shape[0])) - live))
    flat_k[dead] = 0x7FC1
    flat_v[dead] = 0xFFC3
    dirty, _, _, err = run_step(st, torch, k_pool=kp, v_pool=vp)
    assert err == 0
    assert np.array_equal(clean, dirty)


def test_device_error_word_for_bad_slot_and_block():
    st = wl.make_config("tiny")
    shape = shape_of(st)
    import tests.gpu_util as gu
    kp = gu.bf16_dev(st.k_pool, torch)
    vp = gu.bf16_dev(st.v_pool, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, st.num_blocks * st.block_size + 5, -1, 3], dtype=torch.int32,
                         device="cuda")
    bd.paged_kv_write(gu.bf16_dev(st.k_new, torch), gu.bf16_dev(st.v_new, torch), slots, kp, vp,
                      shape, err)
    torch.cuda.synchronize()
    assert int(err.item()) & bd.PA_DEVERR_SLOT
    # a corrupt table entry (outside the pool) reads zeros and raises the block bit
    table = st.block_table.copy()
    table[3, 1] = st.num_blocks + 100
    runner = bd.StepRunner(shape)
    runner.prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    runner.table = torch.from_numpy(table).cuda()
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    runner.attend(gu.bf16_dev(st.q, torch), kp, vp, out)
    torch.cuda.synchronize()
    assert runner.device_error() & bd.PA_DEVERR_BLOCK
    # the other sequences are unaffected
    ref = pa.attention(st.q, pool_np(kp, torch), pool_np(vp, torch), st.block_table,
                       st.cu_seqlens_q, st.ctx_lens, st.Hq)
    o = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_close(o[:3], ref[:3], "unaffected rows")


def test_items_that_break_the_split_rule_are_flagged_and_skipped():
    """A prefill tile's item must cover all of its splits from split 0 and a decode row's item
    exactly one: forged items that do otherwise are skipped with PA_DEVERR_META, and the rows
    of the other items are still right."""
    st = wl.make_step(16, 4, 128, 16, [5000, 4500, 700], [40, 1, 1], seed=91)
    shape = shape_of(st)
    import tests.gpu_util as gu
    kp, vp = gu.bf16_dev(st.k_pool, torch), gu.bf16_dev(st.v_pool, torch)
    q = gu.bf16_dev(st.q, torch)
    ref = pa.attention(st.q, st.k_pool, st.v_pool, st.block_table, st.cu_seqlens_q,
                       st.ctx_lens, st.Hq)
    items = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)
    pre = np.flatnonzero(items["seq"] == 0)
    dec = np.flatnonzero((items["seq"] == 1) & (items["split"] == 0))
    assert np.all(items["n_splits"][pre] == (5000 - 1) // bd.PA_SPLIT_TOKENS + 1) and len(dec) == 4
    for forge in ("prefill_one_split", "prefill_late_start", "decode_two_splits"):
        bad = items.copy()
        if forge == "prefill_one_split":
            bad["n_splits"][pre[0]] = 1
        elif forge == "prefill_late_start":
            bad["split"][pre[0]] = 1
        else:
            bad["n_splits"][dec[0]] = 2
        runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
        runner.items = torch.from_numpy(bad.view(np.int32).reshape(-1).copy()).cuda()
        out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        runner.attend(q, kp, vp, out)
        torch.cuda.synchronize()
        assert runner.device_error() & bd.PA_DEVERR_META, forge
        o = out.view(torch.int16).cpu().numpy().view(np.uint16)
        # sequence 2 (a short decode) has one item, never forged
        assert_close(o[41:42], ref[41:42], forge)


def test_plan_links_that_do_not_move_forward_end_the_list_and_are_flagged():
    """A list link to the item itself, back to an earlier item or past the plan ends that list
    with PA_DEVERR_META; the items of the other lists are still computed right."""
    st = wl.make_step(16, 4, 128, 16, [700, 900, 40] + [300] * 200, [1] * 203, seed=93)
    shape = shape_of(st)
    g = st.Hq // st.Hkv
    import tests.gpu_util as gu
    kp, vp = gu.bf16_dev(st.k_pool, torch), gu.bf16_dev(st.v_pool, torch)
    q = gu.bf16_dev(st.q, torch)
    ref = pa.attention(st.q, st.k_pool, st.v_pool, st.block_table, st.cu_seqlens_q,
                       st.ctx_lens, st.Hq)
    items = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)
    second = int(items["next"][0])                 # list 0's second item
    assert len(items) > bd.PA_PLAN_CTAS and second > 1
    other = list_of(items, 1)                      # list 1 is never forged
    for forge in ("self", "back", "past"):
        bad = items.copy()
        if forge == "self":
            bad["next"][second] = second
        elif forge == "back":
            bad["next"][second] = 1
        else:
            bad["next"][0] = len(items)
        runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
        runner.items = torch.from_numpy(bad.view(np.int32).reshape(-1).copy()).cuda()
        out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        runner.attend(q, kp, vp, out)
        torch.cuda.synchronize()
        assert runner.device_error() & bd.PA_DEVERR_META, forge
        o = out.view(torch.int16).cpu().numpy().view(np.uint16)
        got = np.stack([o[items["q_start"][j], items["kv_head"][j] * g:(items["kv_head"][j] + 1) * g]
                        for j in other])
        want = np.stack([ref[items["q_start"][j], items["kv_head"][j] * g:(items["kv_head"][j] + 1) * g]
                         for j in other])
        assert_close(got, want, forge)


def list_of(items, c):
    """Item indices of list c of a well-formed plan."""
    got, idx = [], c
    while idx >= 0:
        got.append(idx)
        idx = int(items["next"][idx]) if items["next"][idx] > 0 else -1
    return got


def test_host_rejects_bad_arguments_before_launch():
    st = wl.make_config("tiny")
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    import tests.gpu_util as gu
    q = gu.bf16_dev(st.q, torch)
    kp = gu.bf16_dev(st.k_pool, torch)
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.PagedAttnError):
        bd.paged_attention_step(q, kp, kp, runner.table, runner.cu, runner.ctx, 5000,
                                runner.items, None, out, shape)     # needs a workspace
    bad = bd.Shape.make(st.Hq, st.Hkv, 96, st.block_size, st.num_blocks)
    with pytest.raises(bd.PagedAttnError):
        bd.paged_attention_step(q, kp, kp, runner.table, runner.cu, runner.ctx, 100,
                                runner.items, runner.ws, out, bad)


def test_negative_row_start_is_skipped_without_writing_outside_out():
    """cu_seqlens_q forged on the device so that a multi-split decode sequence starts at row
    -1: the attention kernel flags its items (PA_DEVERR_META) and skips them, the split
    combine skips the row, and nothing lands outside `out` (guard rows on both sides)."""
    st = wl.make_step(16, 4, 128, 16, [5000, 4500, 700], [1, 1, 1], seed=94)
    shape = shape_of(st)
    import tests.gpu_util as gu
    kp, vp = gu.bf16_dev(st.k_pool, torch), gu.bf16_dev(st.v_pool, torch)
    q = gu.bf16_dev(st.q, torch)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    cu = st.cu_seqlens_q.copy()
    cu[0], cu[1] = -1, 0                       # sequence 0: one row starting at -1
    runner.cu = torch.from_numpy(cu).cuda()
    guard = torch.full((st.T + 2, st.Hq, st.D), 7.0, dtype=torch.bfloat16, device="cuda")
    out = guard[1:st.T + 1]
    runner.ws.fill_(float("nan"))
    runner.attend(q, kp, vp, out)
    torch.cuda.synchronize()
    assert runner.device_error() & bd.PA_DEVERR_META
    g = guard.float().cpu().numpy()
    assert np.all(g[0] == 7.0) and np.all(g[st.T + 1] == 7.0)


def test_host_rejects_a_misaligned_workspace():
    st = wl.make_step(8, 2, 128, 16, [3000], [1], seed=95)
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    import tests.gpu_util as gu
    q, kp = gu.bf16_dev(st.q, torch), gu.bf16_dev(st.k_pool, torch)
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(runner.ws.numel() + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(bd.PagedAttnError) as e:
        bd.paged_attention_step(q, kp, kp, runner.table, runner.cu, runner.ctx, runner.max_ctx,
                                runner.items, ws[1:], out, shape)
    assert e.value.status == bd.PA_ERR_INVALID


def test_a_wait_that_runs_out_sets_the_timeout_bit_and_the_device_stays_usable():
    """The bounded-wait error path, made to run without faulting anything: the test entry
    point has the softmax role wait 2 ms on a barrier nothing completes. The call returns, the
    error word carries PA_DEVERR_TIMEOUT, and the next ordinary step on the same buffers is
    the oracle's, with a clean error word."""
    for st in (wl.make_config("tiny"), wl.make_step(32, 8, 128, 16, [3000, 40, 700], [1, 1, 64],
                                                    seed=96)):
        shape = shape_of(st)
        import tests.gpu_util as gu
        kp, vp = gu.bf16_dev(st.k_pool, torch), gu.bf16_dev(st.v_pool, torch)
        q = gu.bf16_dev(st.q, torch)
        runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
        runner.write(gu.bf16_dev(st.k_new, torch), gu.bf16_dev(st.v_new, torch), kp, vp)
        out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        ws = runner.ws
        lib = bd.load()
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.paged_attention_step_wait_test(
            q.data_ptr(), kp.data_ptr(), vp.data_ptr(), runner.table.data_ptr(),
            int(runner.table.shape[1]), runner.cu.data_ptr(), runner.ctx.data_ptr(), st.B, st.T,
            runner.max_ctx, runner.items.data_ptr(), int(runner.items.numel() // bd.ITEM_INTS),
            ws.data_ptr() if ws is not None and ws.numel() else None,
            0 if ws is None else ws.numel() * 4, out.data_ptr(), C.byref(shape),
            runner.err.data_ptr(), 2_000_000, stream)
        assert rc == bd.PA_OK
        torch.cuda.synchronize()
        assert runner.device_error() & bd.PA_DEVERR_TIMEOUT
        runner.err.zero_()
        runner.attend(q, kp, vp, out)
        torch.cuda.synchronize()
        assert runner.device_error() == 0
        ref = pa.attention(st.q, pool_np(kp, torch), pool_np(vp, torch), st.block_table,
                           st.cu_seqlens_q, st.ctx_lens, st.Hq)
        assert_close(out.view(torch.int16).cpu().numpy().view(np.uint16), ref, "after a timeout")


def test_wait_test_rejects_limits_outside_its_range():
    st = wl.make_config("tiny")
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    import tests.gpu_util as gu
    q = gu.bf16_dev(st.q, torch)
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    lib = bd.load()
    for never in (0, 2_000_000_000):
        rc = lib.paged_attention_step_wait_test(
            q.data_ptr(), q.data_ptr(), q.data_ptr(), runner.table.data_ptr(),
            int(runner.table.shape[1]), runner.cu.data_ptr(), runner.ctx.data_ptr(), st.B, st.T,
            runner.max_ctx, runner.items.data_ptr(), int(runner.items.numel() // bd.ITEM_INTS), None, 0,
            out.data_ptr(), C.byref(shape), None, never, None)
        assert rc == bd.PA_ERR_INVALID


def test_no_wait_runs_out_silently():
    """Every wait of a step answers long before its one-second limit. The drains at a CTA's end
    give up at that limit without an error bit (the copies and MMAs they wait for are the CTA's
    own), so a barrier that can never complete there (a wrong arrival count, say) would leave
    the outputs right and every launch a second long: timed here, it cannot hide."""
    cases = [wl.make_config("tiny"),
             wl.make_step(32, 8, 128, 16, [3000, 40, 9000, 5000], [1, 1, 512, 1], seed=97),
             wl.make_step(16, 4, 64, 16, [700, 2600], [64, 1], seed=98)]
    for st in cases:
        shape = shape_of(st)
        import tests.gpu_util as gu
        kp, vp = gu.bf16_dev(st.k_pool, torch), gu.bf16_dev(st.v_pool, torch)
        q = gu.bf16_dev(st.q, torch)
        runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
        runner.write(gu.bf16_dev(st.k_new, torch), gu.bf16_dev(st.v_new, torch), kp, vp)
        out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        runner.attend(q, kp, vp, out)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(5):
            runner.attend(q, kp, vp, out)
        ev[1].record()
        torch.cuda.synchronize()
        assert runner.device_error() == 0
        assert ev[0].elapsed_time(ev[1]) / 5 < 50.0, (st.name, ev[0].elapsed_time(ev[1]) / 5)
