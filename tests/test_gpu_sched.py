"""The host scheduler and copy-on-write feeding the device step: every step the scheduler
emits goes through pa_alloc_build_step, paged_kv_write and paged_attention_step, and is
checked against the oracle on the oracle's own copy of the pool (KV bytes bit-exact,
attention within the bf16 tolerance). Block copies of a copy-on-write fork are bit-exact."""
import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, bf16_dev, pool_np

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def test_scheduled_steps_match_the_oracle():
    Hq, Hkv, D, bs = 16, 4, 128, 16
    nb = 96
    rng = np.random.default_rng(31)
    sched = bd.Scheduler(nb, bs, chunk=48, budget=96)
    for i, (p, m) in enumerate([(70, 6), (5, 9), (130, 3), (33, 5), (18, 7)]):
        sched.add(i, p, m)
    sched.add(5, 70, 4, leader=0)                 # shares 4 full blocks of sequence 0
    shape = bd.Shape.make(Hq, Hkv, D, bs, nb)
    k_host = wl.random_bf16(rng, (nb, bs, Hkv, D))
    v_host = wl.random_bf16(rng, (nb, bs, Hkv, D))
    kp, vp = bf16_dev(k_host, torch), bf16_dev(v_host, torch)
    max_blocks = 16
    steps = 0
    while sched.counts()[:2] != (0, 0):
        st = sched.step()
        if not st:
            sched.commit()
            continue
        seqs, n_new, ctx = (np.array(x, np.int32) for x in zip(*st))
        cu, slots, table = sched.allocator.build_step(seqs, ctx, n_new, max_blocks)
        T = int(cu[-1])
        q = wl.random_bf16(rng, (T, Hq, D))
        kn = wl.random_bf16(rng, (T, Hkv, D))
        vn = wl.random_bf16(rng, (T, Hkv, D))
        # device step through the C ABI
        runner = bd.StepRunner(shape).prepare(cu, ctx, table, slot_mapping=slots)
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device="cuda")
        runner.run(bf16_dev(q, torch), bf16_dev(kn, torch), bf16_dev(vn, torch), kp, vp, out)
        torch.cuda.synchronize()
        assert runner.device_error() == 0
        # oracle step on its own pool copy
        want_slots = pa.slot_mapping(table, cu, ctx, bs)
        assert np.array_equal(want_slots.astype(np.int32), slots)
        k_host = pa.kv_write(k_host, kn, want_slots)
        v_host = pa.kv_write(v_host, vn, want_slots)
        assert np.array_equal(pool_np(kp, torch), k_host)
        assert np.array_equal(pool_np(vp, torch), v_host)
        want = pa.attention(q, k_host, v_host, table, cu, ctx, Hq)
        assert_close(out.view(torch.int16).cpu().numpy().view(np.uint16), want, f"step {steps}")
        sched.commit()
        steps += 1
    assert steps > 5 and sched.allocator.num_free == nb


def test_copy_on_write_fork_block_copies_are_bit_exact():
    Hq, Hkv, D, bs, nb = 8, 2, 64, 16, 24
    rng = np.random.default_rng(32)
    alloc = bd.Allocator(nb, bs)
    alloc.admit(0, 40)                            # 3 blocks, the last one partial
    alloc.fork(0, 1)
    alloc.ensure_capacity(1, 45)
    pairs = alloc.cow(1, 40, 5)                   # the shared partial block is replaced
    assert len(pairs) == 1
    shape = bd.Shape.make(Hq, Hkv, D, bs, nb)
    k_host = wl.random_bf16(rng, (nb, bs, Hkv, D))
    v_host = wl.random_bf16(rng, (nb, bs, Hkv, D))
    kp, vp = bf16_dev(k_host, torch), bf16_dev(v_host, torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.paged_copy_blocks(i32_dev(np.array(pairs).reshape(-1)), kp, vp, shape, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for old, new in pairs:
        k_host[new] = k_host[old]
        v_host[new] = v_host[old]
    assert np.array_equal(pool_np(kp, torch), k_host)
    assert np.array_equal(pool_np(vp, torch), v_host)
    # the child writes 5 tokens after its copied prefix; the parent's keys stay untouched
    kn = wl.random_bf16(rng, (5, Hkv, D))
    vn = wl.random_bf16(rng, (5, Hkv, D))
    slots = np.array(alloc.slots(1, 40, 5), np.int32)
    bd.paged_kv_write(bf16_dev(kn, torch), bf16_dev(vn, torch), i32_dev(slots), kp, vp, shape,
                      err)
    torch.cuda.synchronize()
    k_host = pa.kv_write(k_host, kn, slots)
    v_host = pa.kv_write(v_host, vn, slots)
    assert np.array_equal(pool_np(kp, torch), k_host)
    t0, t1 = alloc.table(0), alloc.table(1)
    assert np.array_equal(pa.gather(k_host, t1, 40), pa.gather(k_host, t0, 40))
    # a bad pair is skipped and flagged, nothing else moves
    before = pool_np(kp, torch).copy()
    bd.paged_copy_blocks(i32_dev(np.array([3, nb])), kp, vp, shape, err)
    torch.cuda.synchronize()
    assert int(err.item()) & bd.PA_DEVERR_BLOCK
    assert np.array_equal(pool_np(kp, torch), before)
