"""A step captured once in a CUDA graph and replayed with new metadata gives the same bits as
the same steps launched directly ("Finish RL Training Faster: Bitwise-Consistent,
High-Performance, Agent-Driven", section 4.6: decode runs under CUDA graphs and stays
bitwise consistent). The metadata of every step goes into fixed device buffers (plan padded
with n_q == 0 items, table padded with -1) and the graph reads them at replay."""
import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, attend_with_plan, bf16_dev, pool_np, shape_of

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def _steps(B=24, Hq=32, Hkv=8, D=128, bs=16, seed=21):
    """Two consecutive decode steps of the same B sequences: step 2 has one more token per
    sequence. Tables cover the longer context from the start; the pool is shared."""
    rng = np.random.default_rng(seed)
    ctx2 = rng.integers(100, 5000, size=B).astype(np.int32)
    full = wl.make_step(Hq, Hkv, D, bs, ctx2, np.ones(B, np.int32), seed=seed)
    step1, _ = wl.subset(full, range(B), name="step1")
    step1.ctx_lens = (ctx2 - 1).astype(np.int32)
    step1.q = wl.random_bf16(rng, step1.q.shape)
    step1.k_new = wl.random_bf16(rng, step1.k_new.shape)
    step1.v_new = wl.random_bf16(rng, step1.v_new.shape)
    return step1, full


def _eager(st, kp, vp, q, kn, vn):
    r = bd.StepRunner(shape_of(st)).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    out = torch.empty((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    r.run(q, kn, vn, kp, vp, out)
    torch.cuda.synchronize()
    assert r.device_error() == 0
    return out.view(torch.int16).cpu().numpy()


def test_captured_decode_step_replays_new_metadata_bitwise():
    step1, step2 = _steps()
    kp, vp = bf16_dev(step2.k_pool, torch), bf16_dev(step2.v_pool, torch)
    lim = bd.StepLimits(B=step2.B, T=step2.T, max_blocks=step2.block_table.shape[1],
                        max_ctx=8192)
    runner = bd.StepRunner(shape_of(step2), limits=lim)
    q = torch.empty((step2.T, step2.Hq, step2.D), dtype=torch.bfloat16, device="cuda")
    kn = torch.empty((step2.T, step2.Hkv, step2.D), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    out = torch.empty_like(q)
    runner.prepare(step1.cu_seqlens_q, step1.ctx_lens, step1.block_table)
    runner.capture(q, kn, vn, kp, vp, out)
    for st in (step1, step2, step1):
        # new inputs and metadata into the captured buffers, then one replay
        q.copy_(bf16_dev(st.q, torch))
        kn.copy_(bf16_dev(st.k_new, torch))
        vn.copy_(bf16_dev(st.v_new, torch))
        runner.prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
        runner.replay()
        torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy()
        want = _eager(st, kp, vp, bf16_dev(st.q, torch), bf16_dev(st.k_new, torch),
                      bf16_dev(st.v_new, torch))
        assert runner.device_error() == 0
        assert np.array_equal(got, want)
        # and the replayed step is the oracle's attention over the pool it wrote
        ref = pa.attention(st.q, pool_np(kp, torch), pool_np(vp, torch), st.block_table,
                           st.cu_seqlens_q, st.ctx_lens, st.Hq)
        assert_close(got.view(np.uint16), ref, f"replay ctx max {int(st.ctx_lens.max())}")


def test_captured_mixed_step_equals_direct_launch():
    st = wl.make_step(32, 8, 128, 16, [300, 1800, 2500, 640], [1, 1, 200, 37], seed=22)
    kp, vp = bf16_dev(st.k_pool, torch), bf16_dev(st.v_pool, torch)
    lim = bd.StepLimits(B=st.B, T=st.T, max_blocks=st.block_table.shape[1] + 3, max_ctx=4096)
    runner = bd.StepRunner(shape_of(st), limits=lim)
    q, kn, vn = bf16_dev(st.q, torch), bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch)
    out = torch.empty((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    runner.prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    runner.capture(q, kn, vn, kp, vp, out)
    runner.replay()
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy()
    assert runner.device_error() == 0
    assert np.array_equal(got, _eager(st, kp, vp, q, kn, vn))


def test_captured_fp8_mixed_step_equals_direct_launch():
    """The same over an fp8 cache (float8_e4m3fn codes, per-tensor scales)."""
    from oracle import fp8
    st = wl.make_step(32, 8, 128, 16, [300, 1800, 2500, 640], [1, 1, 200, 37], seed=23)
    scales = (0.0125, 0.0117)
    k8 = torch.from_numpy(fp8.quantize(st.k_pool, scales[0])).cuda()
    v8 = torch.from_numpy(fp8.quantize(st.v_pool, scales[1])).cuda()
    lim = bd.StepLimits(B=st.B, T=st.T, max_blocks=st.block_table.shape[1] + 3, max_ctx=4096)
    runner = bd.StepRunner(shape_of(st), limits=lim, kv_scales=scales)
    q, kn, vn = bf16_dev(st.q, torch), bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch)
    out = torch.empty((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    runner.prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    runner.capture(q, kn, vn, k8, v8, out)
    runner.replay()
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy()
    assert runner.device_error() == 0
    eager = bd.StepRunner(shape_of(st), kv_scales=scales).prepare(st.cu_seqlens_q, st.ctx_lens,
                                                                  st.block_table)
    out2 = torch.empty_like(out)
    eager.run(q, kn, vn, k8, v8, out2)
    torch.cuda.synchronize()
    assert eager.device_error() == 0
    assert np.array_equal(got, out2.view(torch.int16).cpu().numpy())


def test_limits_are_enforced_on_the_host():
    st = wl.make_step(8, 2, 64, 16, [40, 50], [1, 1], seed=23)
    lim = bd.StepLimits(B=2, T=2, max_blocks=st.block_table.shape[1], max_ctx=45)
    runner = bd.StepRunner(shape_of(st), limits=lim)
    with pytest.raises(ValueError):
        runner.prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)    # ctx 50 > 45


@pytest.mark.parametrize("name,kv", [("decode", "bf16"), ("mixed", "bf16"), ("prefill", "bf16"),
                                     ("decode", "fp8")])
def test_full_size_bench_graphs_equal_direct_launches(name, kv):
    """The timed configuration of bench.py (its full-size workloads, captured write and
    attention graphs over the padded plan of a StepLimits runner) gives the bits of direct
    launches, which the sampled full-size parity tests compare with the oracle."""
    import bench
    st = bench.make_workload(name, 0)
    g = bench.GpuStep(st, torch, bd, kv=kv)
    g.g_write.replay()
    g.g_attend.replay()
    torch.cuda.synchronize()
    assert g.graph_runner.device_error() == 0
    got = g.out.view(torch.int16).cpu().numpy()
    r = bd.StepRunner(g.shape, kv_scales=g.kv_scales).prepare(st.cu_seqlens_q, st.ctx_lens,
                                                              st.block_table)
    out = torch.empty_like(g.out)
    r.run(g.q, g.kn, g.vn, g.kp, g.vp, out)
    torch.cuda.synchronize()
    assert r.device_error() == 0
    assert np.array_equal(got, out.view(torch.int16).cpu().numpy())
    # the end-to-end pipeline (host metadata, pinned uploads, its own captured graphs), three
    # steps in a row so that both of its buffer sets serve
    evs = [g.submit_e2e(i) for i in range(3)]
    for ev in evs:
        ev.synchronize()
    assert g.pipe.device_error() == 0
    for h in g.h_out:
        assert np.array_equal(h.numpy(), got)
    # the replayed graphs against the oracle on sampled rows (the longest row, both ends of
    # every prefill segment, a seeded sample)
    rng = np.random.default_rng(99)
    rows = set(rng.choice(st.T, size=min(12, st.T), replace=False).tolist())
    rows.add(int(st.cu_seqlens_q[int(np.argmax(st.ctx_lens)) + 1]) - 1)
    for s in range(st.B):
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        if b - a > 1:
            rows.update([a, b - 1])
    rows = np.array(sorted(rows))
    # the oracle reads a compact pool of the blocks those rows' sequences use
    seq_of = np.searchsorted(st.cu_seqlens_q, rows, side="right") - 1
    nblk = (st.ctx_lens + st.block_size - 1) // st.block_size
    used = np.unique(np.concatenate([st.block_table[s, :nblk[s]] for s in np.unique(seq_of)]))
    remap = np.full(st.num_blocks, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    table = np.where(st.block_table >= 0, remap[np.maximum(st.block_table, 0)], -1)
    if kv == "fp8":
        from oracle import fp8
        kp = fp8.dequantize(g.kp.cpu().numpy()[used], g.kv_scales[0])
        vp = fp8.dequantize(g.vp.cpu().numpy()[used], g.kv_scales[1])
    else:
        kp, vp = pool_np(g.kp, torch)[used], pool_np(g.vp, torch)[used]
    ref = pa.attention_rows(st.q, kp, vp, table, st.cu_seqlens_q, st.ctx_lens, st.Hq, rows)
    assert_close(got.view(np.uint16)[rows], ref, f"bench graphs {name} {kv}")


def test_pipeline_of_different_steps_equals_direct_launches():
    """StepPipeline (two buffer sets, host work and copies of one step overlapping the kernels of
    the previous one) gives every step of a stream the bits of direct launches, and the oracle's
    attention."""
    step1, step2 = _steps(seed=31)
    kp, vp = bf16_dev(step2.k_pool, torch), bf16_dev(step2.v_pool, torch)
    lim = bd.StepLimits(B=step2.B, T=step2.T, max_blocks=step2.block_table.shape[1], max_ctx=8192)
    pipe = bd.StepPipeline(shape_of(step2), lim, kp, vp)
    pin = lambda a: torch.from_numpy(a.view(np.int16).copy()).pin_memory()
    stream = [step1, step2, step1, step2, step2]
    host = [(pin(st.q), pin(st.k_new), pin(st.v_new),
             torch.empty((st.T, st.Hq, st.D), dtype=torch.int16).pin_memory()) for st in stream]
    events = [pipe.submit(st.cu_seqlens_q, st.ctx_lens, st.block_table, *h)
              for st, h in zip(stream, host)]
    for ev in events:
        ev.synchronize()
    assert pipe.device_error() == 0
    for st, h in zip(stream, host):
        want = _eager(st, kp, vp, bf16_dev(st.q, torch), bf16_dev(st.k_new, torch),
                      bf16_dev(st.v_new, torch))
        assert np.array_equal(h[3].numpy(), want)
    ref = pa.attention(step2.q, pool_np(kp, torch), pool_np(vp, torch), step2.block_table,
                       step2.cu_seqlens_q, step2.ctx_lens, step2.Hq)
    assert_close(host[-1][3].numpy().view(np.uint16), ref, "pipeline")


def test_pipeline_runs_prefix_shared_steps():
    """Two consecutive decode steps of samples that share their prompts' blocks, through
    StepPipeline (which plans with GROUP / RESUME items): each step's output has the bits of the
    same step planned with plain items only, and the second matches the oracle."""
    full = wl.make_prefix_step(32, 8, 128, 16, prompts=3, samples=6, prompt_tokens=768,
                               cont_max=2600, seed=41)
    rng = np.random.default_rng(42)
    step1, _ = wl.subset(full, range(full.B), name="step1")
    step1.ctx_lens = (full.ctx_lens - 1).astype(np.int32)
    step1.q = wl.random_bf16(rng, step1.q.shape)
    step1.k_new = wl.random_bf16(rng, step1.k_new.shape)
    step1.v_new = wl.random_bf16(rng, step1.v_new.shape)
    shape = shape_of(full)
    for st in (step1, full):
        items = bd.pa_plan_step_shared(shape, st.cu_seqlens_q, st.ctx_lens, st.block_table)
        assert np.sum(items["kind"] == bd.PA_ITEM_GROUP) == 3 * full.Hkv
    kp, vp = bf16_dev(full.k_pool, torch), bf16_dev(full.v_pool, torch)
    lim = bd.StepLimits(B=full.B, T=full.T, max_blocks=full.block_table.shape[1],
                        max_ctx=int(full.ctx_lens.max()))
    pipe = bd.StepPipeline(shape, lim, kp, vp)
    pin = lambda a: torch.from_numpy(a.view(np.int16).copy()).pin_memory()
    host = [(pin(st.q), pin(st.k_new), pin(st.v_new),
             torch.empty((st.T, st.Hq, st.D), dtype=torch.int16).pin_memory())
            for st in (step1, full)]
    events = [pipe.submit(st.cu_seqlens_q, st.ctx_lens, st.block_table, *h)
              for st, h in zip((step1, full), host)]
    for ev in events:
        ev.synchronize()
    assert pipe.device_error() == 0
    # the second step's write lands past the first step's keys, so the final pools serve both
    for st, h in zip((step1, full), host):
        plain = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)
        assert np.array_equal(h[3].numpy(), attend_with_plan(st, kp, vp, plain, torch)), st.name
    ref = pa.attention(full.q, pool_np(kp, torch), pool_np(vp, torch), full.block_table,
                       full.cu_seqlens_q, full.ctx_lens, full.Hq)
    assert_close(host[-1][3].numpy().view(np.uint16), ref, "pipeline, prefix-shared")
