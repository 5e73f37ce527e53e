"""GPU parity of the FP8 KV cache through the C ABI ("P3: native paged-KV continuous-batching
sampler", Review, kv_dtype item; "Finish RL Training Faster: Bitwise-Consistent, ...", 4.2):
write codes bit-exact against oracle/fp8.py, attention within the bf16 tolerance of the fp64
oracle over the dequantised pools (code * scale), and bit identity across batch mixes and
between prefill and decode within the fp8 path."""
import numpy as np
import pytest

import oracle.paged_attention as pa
from oracle import fp8
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, bf16_dev, shape_of

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    build.build()
    return bd.load()


def scales_for(st):
    """Per-tensor scales from the data the step holds (amax / 448, fp32)."""
    ks = float(np.float32(np.abs(pa.bf16_to_f64(st.k_pool)).max() / 448.0))
    vs = float(np.float32(np.abs(pa.bf16_to_f64(st.v_pool)).max() / 448.0))
    return ks, vs


def u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def run_fp8(st, kcodes, vcodes, ks, vs, write=True):
    """fp8 write + attention on the device; returns (out uint16, k codes, v codes, err)."""
    shape = shape_of(st)
    runner = bd.StepRunner(shape, kv_scales=(ks, vs)).prepare(st.cu_seqlens_q, st.ctx_lens,
                                                              st.block_table)
    kp, vp = u8_dev(kcodes), u8_dev(vcodes)
    out = torch.full((st.T, st.Hq, st.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    if write and st.T > 0:
        runner.write(bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch), kp, vp)
    runner.attend(bf16_dev(st.q, torch), kp, vp, out)
    torch.cuda.synchronize()
    o = out.view(torch.int16).cpu().numpy().view(np.uint16)
    return o, kp.cpu().numpy(), vp.cpu().numpy(), runner.device_error()


def oracle_fp8(st, ks, vs):
    """Codes of the pools before the step (quantised bf16 pools), the codes after the step's
    write, and the fp64 attention over the dequantised pools."""
    k0, v0 = fp8.quantize(st.k_pool, ks), fp8.quantize(st.v_pool, vs)
    slots = pa.slot_mapping(st.block_table, st.cu_seqlens_q, st.ctx_lens, st.block_size)
    k1 = pa.kv_write(k0, fp8.quantize(st.k_new, ks), slots)
    v1 = pa.kv_write(v0, fp8.quantize(st.v_new, vs), slots)
    out = pa.attention(st.q, fp8.dequantize(k1, ks), fp8.dequantize(v1, vs), st.block_table,
                       st.cu_seqlens_q, st.ctx_lens, st.Hq)
    return k0, v0, k1, v1, out


MID_CTX = [1, 17, 127, 128, 129, 1023, 1024, 1025, 2047, 2048, 2049, 4097, 200, 2100, 4200, 5, 384]
MID_NQ = [1] * 12 + [200, 77, 33, 5, 129]


@pytest.mark.parametrize("Hq,Hkv,bs", [(32, 8, 16), (8, 8, 32), (64, 8, 64), (16, 1, 128),
                                       (32, 8, 8), (64, 4, 16), (32, 2, 128)])
def test_fp8_mixed_step_all_rows(Hq, Hkv, bs):
    st = wl.make_step(Hq, Hkv, 128, bs, MID_CTX, MID_NQ, seed=Hq * 11 + bs)
    ks, vs = scales_for(st)
    k0, v0, k1, v1, ref = oracle_fp8(st, ks, vs)
    out, kc, vc, err = run_fp8(st, k0, v0, ks, vs)
    assert err == 0
    assert np.array_equal(kc, k1) and np.array_equal(vc, v1)        # write: bit-exact codes
    assert_close(out, ref, f"fp8 Hq{Hq} Hkv{Hkv} bs{bs}")


@pytest.mark.parametrize("name", ["decode", "mixed"])
def test_fp8_full_size_workloads_sampled(name):
    st = wl.make_config(name)
    ks, vs = scales_for(st)
    k0, v0 = fp8.quantize(st.k_pool, ks), fp8.quantize(st.v_pool, vs)
    out, kc, vc, err = run_fp8(st, k0, v0, ks, vs)
    assert err == 0
    slots = pa.slot_mapping(st.block_table, st.cu_seqlens_q, st.ctx_lens, st.block_size)
    flat = kc.reshape(-1, st.Hkv, st.D)
    assert np.array_equal(flat[slots], fp8.quantize(st.k_new, ks))
    # a sample of sequences (the longest, every prefill segment, a few others); the oracle
    # runs on a compact pool of their blocks only
    rng = np.random.default_rng(5)
    n_q = np.diff(st.cu_seqlens_q)
    seqs = set(rng.choice(st.B, size=min(6, st.B), replace=False).tolist())
    seqs |= {int(np.argmax(st.ctx_lens))} | set(np.flatnonzero(n_q > 1).tolist())
    seqs = sorted(seqs)
    nblk = (st.ctx_lens + st.block_size - 1) // st.block_size
    used = np.unique(np.concatenate([st.block_table[s, :nblk[s]] for s in seqs]))
    remap = {int(b): i for i, b in enumerate(used)}
    sub, rows = wl.subset(st, seqs)
    table = np.array([[remap.get(int(b), 0) if j < nblk[s] else -1
                       for j, b in enumerate(st.block_table[s])] for s in seqs], dtype=np.int32)
    rows = np.concatenate(rows)
    pick = np.unique(np.concatenate([rng.choice(len(rows), size=min(24, len(rows)), replace=False),
                                     sub.cu_seqlens_q[1:] - 1, sub.cu_seqlens_q[:-1]]))
    ref = pa.attention_rows(sub.q, fp8.dequantize(kc[used], ks), fp8.dequantize(vc[used], vs),
                            table, sub.cu_seqlens_q, sub.ctx_lens, st.Hq, pick)
    assert_close(out[rows[pick]], ref, f"fp8 {name}")


def test_fp8_prefill_equals_decode_bitwise():
    """The last m tokens of a sequence as one prefill chunk, and as m decode rows over the same
    fp8 cache: equal bits."""
    L, m = 3000, 300
    st = wl.make_step(32, 8, 128, 16, [L], [m], seed=L + m)
    ks, vs = scales_for(st)
    k0, v0 = fp8.quantize(st.k_pool, ks), fp8.quantize(st.v_pool, vs)
    pre, kc, vc, _ = run_fp8(st, k0, v0, ks, vs)
    ctx = np.arange(L - m + 1, L + 1, dtype=np.int32)
    dec = wl.Step(name="dec", Hq=32, Hkv=8, D=128, block_size=16, num_blocks=st.num_blocks,
                  ctx_lens=ctx, n_q=np.ones(m, np.int32),
                  cu_seqlens_q=np.arange(m + 1, dtype=np.int32),
                  block_table=np.repeat(st.block_table, m, axis=0), q=st.q,
                  k_new=st.k_new, v_new=st.v_new, k_pool=st.k_pool, v_pool=st.v_pool)
    out, _, _, _ = run_fp8(dec, kc, vc, ks, vs, write=False)
    assert np.array_equal(out, pre)


def test_fp8_alone_vs_among_others_bitwise():
    ctx = [3000, 17, 2070, 2049, 128, 700, 4100, 64]
    nq = [1, 1, 40, 1, 128, 1, 1, 64]
    st = wl.make_step(32, 8, 128, 16, ctx, nq, seed=23)
    ks, vs = scales_for(st)
    k0, v0 = fp8.quantize(st.k_pool, ks), fp8.quantize(st.v_pool, vs)
    full, kc, vc, _ = run_fp8(st, k0, v0, ks, vs)
    for s in range(st.B):
        sub, _ = wl.subset(st, [s], st.k_pool, st.v_pool)
        got, _, _, _ = run_fp8(sub, kc, vc, ks, vs, write=False)
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        assert np.array_equal(got, full[a:b]), f"seq {s}"


def test_fp8_host_rejects_bad_arguments():
    st = wl.make_config("tiny")                      # head_dim 64: not supported by the fp8 path
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    q = bf16_dev(st.q, torch)
    pool = torch.zeros(st.k_pool.shape, dtype=torch.uint8, device="cuda")
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.PagedAttnError):
        bd.paged_attention_step_fp8(q, pool, pool, runner.table, runner.cu, runner.ctx, 128,
                                    runner.items, 1.0, 1.0, runner.ws, out, shape)
    st = wl.make_step(16, 4, 128, 16, [40], [1], seed=3)
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    pool = torch.zeros(st.k_pool.shape, dtype=torch.uint8, device="cuda")
    q = bf16_dev(st.q, torch)
    out = torch.zeros((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(bd.PagedAttnError):
            bd.paged_attention_step_fp8(q, pool, pool, runner.table, runner.cu, runner.ctx, 40,
                                        runner.items, bad, 1.0, runner.ws, out, shape)
        with pytest.raises(bd.PagedAttnError):
            bd.paged_kv_write_fp8(bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch),
                                  runner.slots, pool, pool, 1.0, bad, shape)
