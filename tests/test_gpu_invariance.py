"""Bitwise invariance of the GPU path: a sequence's output bits do not depend on the batch
around it, on prefill vs decode, or on where its blocks sit in the pool ("P3: native
paged-KV continuous-batching sampler", Evidence item 2 and the kernel contract in Design /
paged.py; "Finish RL Training Faster: Bitwise-Consistent, High-Performance, Agent-Driven",
section 2: batch independence and phase consistency)."""
import numpy as np
import pytest

from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import attend_with_plan, pool_np, run_step

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def sub_step(st: wl.Step, idx, k_pool, v_pool):
    """A step made of sequences `idx` of st (same tables, same pool, same rows)."""
    return wl.subset(st, list(idx), k_pool, v_pool)


def test_alone_vs_among_others():
    """Each sequence alone, and among 1, 3 and 7 others in shuffled orders: equal bits."""
    ctx = [3000, 17, 2070, 2049, 128, 700, 4100, 64, 2048, 999]
    nq = [1, 1, 40, 1, 128, 1, 1, 64, 1, 300]
    st = wl.make_step(32, 8, 128, 16, ctx, nq, seed=21)
    full, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    rng = np.random.default_rng(5)
    for s in range(st.B):
        for n_others in (0, 1, 3, 7):
            others = rng.choice([i for i in range(st.B) if i != s], size=n_others, replace=False)
            idx = list(others) + [s]
            rng.shuffle(idx)
            sub, rows = sub_step(st, idx, kpn, vpn)
            out, _, _, _ = run_step(sub, torch, write=False)
            j = idx.index(s)
            got = out[sub.cu_seqlens_q[j]:sub.cu_seqlens_q[j + 1]]
            want = full[rows[j]]
            assert np.array_equal(got, want), f"seq {s} among {n_others} others"


@pytest.mark.parametrize("Hq,Hkv,D,bs,L,m", [(32, 8, 128, 16, 2600, 300),
                                              (64, 8, 128, 32, 1200, 140),
                                              (8, 4, 64, 16, 900, 200)])
def test_prefill_equals_decode(Hq, Hkv, D, bs, L, m):
    """The last m tokens of a sequence as one prefill chunk, and as m separate decode rows
    over the same cache (one per position, each with its own ctx): equal bits."""
    st = wl.make_step(Hq, Hkv, D, bs, [L], [m], seed=L + m)
    pre, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    ctx = np.arange(L - m + 1, L + 1, dtype=np.int32)
    dec = wl.Step(name="dec", Hq=Hq, Hkv=Hkv, D=D, block_size=bs, num_blocks=st.num_blocks,
                  ctx_lens=ctx, n_q=np.ones(m, np.int32),
                  cu_seqlens_q=np.arange(m + 1, dtype=np.int32),
                  block_table=np.repeat(st.block_table, m, axis=0), q=st.q,
                  k_new=st.k_new, v_new=st.v_new, k_pool=kpn, v_pool=vpn)
    out, _, _, _ = run_step(dec, torch, write=False)
    assert np.array_equal(out, pre)


def test_chunking_does_not_change_bits():
    """One 513-row chunk vs the same rows split into chunks of 1, 7, 128 and 250 rows that
    run as separate steps over the same cache."""
    L = 1900
    st = wl.make_step(32, 8, 128, 16, [L], [513], seed=99)
    whole, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    for chunk in (1, 7, 128, 250):
        got = []
        start = L - 513
        while start < L:
            n = min(chunk, L - start)
            rows = np.arange(start - (L - 513), start - (L - 513) + n)
            s = wl.Step(name="chunk", Hq=32, Hkv=8, D=128, block_size=16,
                        num_blocks=st.num_blocks, ctx_lens=np.array([start + n], np.int32),
                        n_q=np.array([n], np.int32), cu_seqlens_q=np.array([0, n], np.int32),
                        block_table=st.block_table, q=st.q[rows], k_new=st.k_new[rows],
                        v_new=st.v_new[rows], k_pool=kpn, v_pool=vpn)
            o, _, _, _ = run_step(s, torch, write=False)
            got.append(o)
            start += n
        assert np.array_equal(np.concatenate(got), whole), f"chunk {chunk}"


def test_block_renaming_gives_equal_bits():
    st = wl.make_step(32, 8, 128, 16, [2500, 33, 1030], [1, 33, 5], seed=31,
                      num_blocks=400)
    a, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    perm = np.random.default_rng(2).permutation(st.num_blocks)
    kp2 = np.empty_like(kpn)
    vp2 = np.empty_like(vpn)
    kp2[perm] = kpn
    vp2[perm] = vpn
    t2 = np.where(st.block_table >= 0, perm[np.maximum(st.block_table, 0)], -1).astype(np.int32)
    st2 = wl.Step(name="perm", Hq=32, Hkv=8, D=128, block_size=16, num_blocks=st.num_blocks,
                  ctx_lens=st.ctx_lens, n_q=st.n_q, cu_seqlens_q=st.cu_seqlens_q, block_table=t2,
                  q=st.q, k_new=st.k_new, v_new=st.v_new, k_pool=kp2, v_pool=vp2)
    b, _, _, _ = run_step(st2, torch, write=False)
    assert np.array_equal(a, b)


def test_longtail_rerun_each_sequence_alone():
    """The long-tail rollout decode workload: every sequence re-run alone gives the bits it
    got inside the 128-row batch."""
    st = wl.make_config("longtail")
    full, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    for s in range(st.B):
        sub, rows = sub_step(st, [s], kpn, vpn)
        out, _, _, _ = run_step(sub, torch, write=False)
        assert np.array_equal(out, full[rows[0]]), f"sequence {s}"


def test_repeat_runs_are_bitwise_deterministic():
    st = wl.make_config("mixed")
    a, kp, vp, _ = run_step(st, torch)
    kpn, vpn = pool_np(kp, torch), pool_np(vp, torch)
    st.k_pool, st.v_pool = kpn, vpn
    b, _, _, _ = run_step(st, torch, write=False)
    c, _, _, _ = run_step(st, torch, write=False)
    assert np.array_equal(a, b) and np.array_equal(b, c)


def test_prefix_groups_give_the_bits_of_plain_items():
    """Samples that share a prompt's blocks, planned with GROUP / RESUME items (the shared tiles
    read once for all of them, each row's softmax state carried across) and with PLAIN items
    only: equal bits for every row, also for a sample run alone."""
    st = wl.make_config("prefix")
    sub, _ = wl.subset(st, range(32))                 # 4 prompts x 8 samples
    shape = bd.Shape.make(sub.Hq, sub.Hkv, sub.D, sub.block_size, sub.num_blocks)
    out, kp, vp, err = run_step(sub, torch)           # the runner plans with sharing
    assert err == 0
    shared = bd.pa_plan_step_shared(shape, sub.cu_seqlens_q, sub.ctx_lens, sub.block_table)
    assert np.sum(shared["kind"] == bd.PA_ITEM_GROUP) == 4 * sub.Hkv
    plain = bd.pa_plan_step(shape, sub.cu_seqlens_q, sub.ctx_lens)
    got_shared = attend_with_plan(sub, kp, vp, shared, torch)
    got_plain = attend_with_plan(sub, kp, vp, plain, torch)
    assert np.array_equal(got_shared, got_plain)
    assert np.array_equal(out.view(np.int16), got_plain)
    # a sample alone (no group at all) and a group of two
    for idx in ([13], [16, 17]):
        one, rows = wl.subset(sub, idx)
        items = bd.pa_plan_step_shared(shape, one.cu_seqlens_q, one.ctx_lens, one.block_table)
        assert np.sum(items["kind"] == bd.PA_ITEM_GROUP) == (sub.Hkv if len(idx) == 2 else 0)
        alone = attend_with_plan(one, kp, vp, items, torch)
        assert np.array_equal(alone, got_plain[np.concatenate(rows)])
