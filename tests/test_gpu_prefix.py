"""Prefix sharing on the GPU: steps whose samples share a prompt's blocks, planned with GROUP /
RESUME items (each shared tile read once for the whole group, every row's softmax state carried
from the GROUP item to its RESUME item) give the bits of the same step planned with plain items
only, and stay within the tolerance of the fp64 oracle. Cases cover head_dim 64 and 128, block
sizes 16 to 64, one, four, eight and sixteen q heads per KV head, groups up to the 128-row
limit (and a prompt with more samples than one group holds), prompts that are not a whole
number of blocks, rows past the first split (their later splits are plain items, folded by the
combine), and an fp8 cache."""
import numpy as np
import pytest

import oracle.fp8 as fp8
import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, attend_with_plan, bf16_dev, pool_np, run_step, shape_of

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def groups_of(st):
    items = bd.pa_plan_step_shared(shape_of(st), st.cu_seqlens_q, st.ctx_lens, st.block_table)
    return items[items["kind"] == bd.PA_ITEM_GROUP]


# (Hq, Hkv, D, block_size, prompts, samples, prompt tokens, continuation max, seed)
CASES = [
    (32, 8, 128, 16, 3, 5, 640, 2500, 201),     # 5 shared tiles, some rows past 2048 keys
    (16, 4, 64, 32, 2, 40, 256, 1500, 202),     # 40 samples: groups of 32 (the row limit) + 8
    (8, 8, 128, 64, 2, 3, 1920, 3000, 203),     # g = 1, 15 shared tiles (the most split 0 holds)
    (16, 2, 64, 16, 4, 2, 300, 700, 204),       # g = 8; 18 whole blocks = 2 whole tiles shared
    (16, 1, 128, 16, 2, 10, 512, 900, 206),     # g = 16: a group of 8 fills a tile's 128 rows
]


@pytest.mark.parametrize("case", CASES, ids=[f"D{c[2]}-bs{c[3]}-g{c[0] // c[1]}" for c in CASES])
def test_shared_plan_equals_plain_plan_and_oracle(case):
    Hq, Hkv, D, bs, P, G, prompt, cont, seed = case
    st = wl.make_prefix_step(Hq, Hkv, D, bs, prompts=P, samples=G, prompt_tokens=prompt,
                             cont_max=cont, seed=seed)
    groups = groups_of(st)
    assert len(groups) >= P * Hkv and np.all(groups["tile0"] >= 2)
    assert np.all(groups["n_q"] * (Hq // Hkv) <= 128)       # a tile holds 128 rows
    out, kp, vp, err = run_step(st, torch)        # the runner plans with sharing
    assert err == 0
    plain = bd.pa_plan_step(shape_of(st), st.cu_seqlens_q, st.ctx_lens)
    assert np.array_equal(out.view(np.int16), attend_with_plan(st, kp, vp, plain, torch))
    ref = pa.attention(st.q, pool_np(kp, torch), pool_np(vp, torch), st.block_table,
                       st.cu_seqlens_q, st.ctx_lens, st.Hq)
    assert_close(out, ref, f"prefix {case}")


def test_shared_plan_over_an_fp8_cache():
    st = wl.make_prefix_step(32, 8, 128, 16, prompts=2, samples=6, prompt_tokens=512,
                             cont_max=2400, seed=205)
    assert len(groups_of(st)) == 2 * 8
    ks = float(np.float32(np.abs(pa.bf16_to_f64(st.k_pool)).max() / 448.0))
    vs = float(np.float32(np.abs(pa.bf16_to_f64(st.v_pool)).max() / 448.0))
    shape = shape_of(st)
    dev8 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()
    kp, vp = dev8(fp8.quantize(st.k_pool, ks)), dev8(fp8.quantize(st.v_pool, vs))
    runner = bd.StepRunner(shape, kv_scales=(ks, vs)).prepare(st.cu_seqlens_q, st.ctx_lens,
                                                              st.block_table)
    runner.write(bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch), kp, vp)
    q = bf16_dev(st.q, torch)
    out = torch.full((st.T, st.Hq, st.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    runner.attend(q, kp, vp, out)
    torch.cuda.synchronize()
    assert runner.device_error() == 0
    shared_bits = out.view(torch.int16).cpu().numpy()
    # the same step with plain items only
    plain = bd.pa_plan_step(shape, st.cu_seqlens_q, st.ctx_lens)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    max_ctx = int(st.ctx_lens.max())
    ws = torch.empty((bd.pa_workspace_bytes(shape, st.T, max_ctx) + 3) // 4, dtype=torch.float32,
                     device="cuda")
    out2 = torch.full_like(out, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.paged_attention_step_fp8(q, kp, vp, dev(st.block_table), dev(st.cu_seqlens_q),
                                dev(st.ctx_lens), max_ctx, dev(plain.view(np.int32).reshape(-1)),
                                ks, vs, ws, out2, shape, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(shared_bits, out2.view(torch.int16).cpu().numpy())
    # and the oracle over the dequantised codes the write left
    k1, v1 = kp.cpu().numpy(), vp.cpu().numpy()
    ref = pa.attention(st.q, fp8.dequantize(k1, ks), fp8.dequantize(v1, vs), st.block_table,
                       st.cu_seqlens_q, st.ctx_lens, st.Hq)
    assert_close(shared_bits.view(np.uint16), ref, "prefix over fp8")
