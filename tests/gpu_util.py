"""Helpers for the GPU tests: run one step through the C ABI and compare with the oracle."""
import numpy as np

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl

MAX_ABS = 1.5e-2      # tolerance on bf16 outputs vs the fp64 oracle (max |diff|)
MEAN_ABS = 2e-3       # and mean |diff|


def to_dev(a, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(a, torch):
    return to_dev(a.view(np.int16), torch).view(torch.bfloat16)


def shape_of(st: wl.Step) -> bd.Shape:
    return bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)


def run_step(st: wl.Step, torch, k_pool=None, v_pool=None, write=True):
    """kv_write + attention on the device. Returns (out uint16 [T,Hq,D], k_pool, v_pool as
    uint16 numpy, device error word)."""
    shape = shape_of(st)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    kp = bf16_dev(st.k_pool if k_pool is None else k_pool, torch)
    vp = bf16_dev(st.v_pool if v_pool is None else v_pool, torch)
    q = bf16_dev(st.q, torch)
    out = torch.full((st.T, st.Hq, st.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    if write and st.T > 0:
        runner.write(bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch), kp, vp)
    runner.attend(q, kp, vp, out)
    torch.cuda.synchronize()
    o = out.view(torch.int16).cpu().numpy().view(np.uint16)
    return o, kp, vp, runner.device_error()


def pool_np(t, torch):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close(got_bits: np.ndarray, want: np.ndarray, what: str = ""):
    got = pa.bf16_to_f64(got_bits)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - want)
    assert d.max() <= MAX_ABS, f"{what}: max|diff| {d.max():.3e}"
    assert d.mean() <= MEAN_ABS, f"{what}: mean|diff| {d.mean():.3e}"
    return float(d.max()), float(d.mean())
