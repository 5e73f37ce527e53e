"""Helpers for the GPU tests: run one step through the C ABI and compare with the oracle."""
import numpy as np

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl

MAX_ABS = 1.5e-2      # tolerance on bf16 outputs vs the fp64 oracle (max |diff|)
MEAN_ABS = 2e-3       # and mean |diff|
# Scaled to each (row, head): max_d |diff| <= REL * rms_d(oracle row) + REL_FLOOR. The absolute
# bounds above cannot see a dropped key tile at long context (outputs there are only ~0.01
# RMS); this one can. The kernel rounds P to bf16 (2^-9 relative), sums l from the fp32 P and
# rounds the output to bf16 (2^-9 relative), which an fp32 emulation puts at <= 2^-6.4 of the
# row's RMS; a dropped 128-key tile moves a row by >= 0.08 of its RMS at ctx <= 40960
# (tests/test_oracle_pins.py checks that on the oracle).
REL = 2.0 ** -5
REL_FLOOR = 1e-4


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


def rel_error(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Per (row, head): max_d |got - want| / (REL * rms_d(want) + REL_FLOOR); <= 1 passes."""
    d = np.abs(got - want).max(axis=-1)
    rms = np.sqrt((want ** 2).mean(axis=-1))
    return d / (REL * rms + REL_FLOOR)


# (what, max|diff|, mean|diff|, max scaled ratio) of every comparison in this process; the
# test session writes them to the file PA_PARITY_STATS names, if set
STATS = []


def assert_close(got_bits: np.ndarray, want: np.ndarray, what: str = ""):
    """bf16 output bits against the fp64 oracle [rows, Hq, D]: the absolute bounds and the
    per-(row, head) scaled bound. Returns (max|diff|, mean|diff|, max scaled ratio)."""
    got = pa.bf16_to_f64(got_bits)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - want)
    assert d.max() <= MAX_ABS, f"{what}: max|diff| {d.max():.3e}"
    assert d.mean() <= MEAN_ABS, f"{what}: mean|diff| {d.mean():.3e}"
    r = rel_error(got, want) if d.size else np.zeros(1)
    if d.size:
        STATS.append((what, float(d.max()), float(d.mean()), float(r.max())))
    worst = np.unravel_index(int(np.argmax(r)), r.shape) if d.size else ()
    assert r.max() <= 1.0, (f"{what}: (row, head) {worst} off by {r.max():.2f} x "
                            f"(REL * rms + floor)")
    return float(d.max()), float(d.mean()), float(r.max())


def attend_with_plan(st, kp, vp, items, torch):
    """Attention of step st over pools kp / vp (already written) with a given plan."""
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = dev(st.q.view(np.int16)).view(torch.bfloat16)
    out = torch.full((st.T, st.Hq, st.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    max_ctx = int(st.ctx_lens.max())
    ws = torch.empty((bd.pa_workspace_bytes(shape, st.T, max_ctx) + 3) // 4, dtype=torch.float32,
                     device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.paged_attention_step(q, kp, vp, dev(st.block_table), dev(st.cu_seqlens_q),
                            dev(st.ctx_lens), max_ctx,
                            dev(items.view(np.int32).reshape(-1)), ws, out, shape, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.view(torch.int16).cpu().numpy()
