"""The allocation-free attention entry point (paged_attention_step_static_scratch).

It exists for callers that may not allocate device memory while they run a step (memory
reserved up front by a serving process, a plug-in that only gets tensors from its host
framework, a loop that cannot take cudaMalloc's implicit synchronisation): it keeps its split
partials in a fixed array inside the library instead of a caller-provided workspace. This
test calls it through the C ABI, twice in a row with different steps that both need the
scratch, and checks that each output has the bits of paged_attention_step's (the same
kernels with the same arithmetic; only where the partials live differs), and that the call
leaves the device's free memory unchanged. It also checks that a step too large for the
fixed array is refused. This file is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import binding as bd
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import MAX_ABS, MEAN_ABS, bf16_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

STATIC_SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from continuous_batching_gb300 import build
    build.build()
    lib = bd.load()
    f = lib.paged_attention_step_static_scratch
    f.restype = C.c_int32
    vp = C.c_void_p
    f.argtypes = [vp, vp, vp, vp, C.c_int32, vp, vp, C.c_int32, C.c_int32, C.c_int32, vp,
                  C.c_int32, vp, C.POINTER(bd.Shape), vp, vp]
    return lib


def _prepare(st):
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    runner = bd.StepRunner(shape).prepare(st.cu_seqlens_q, st.ctx_lens, st.block_table)
    kp, vp = bf16_dev(st.k_pool, torch), bf16_dev(st.v_pool, torch)
    runner.write(bf16_dev(st.k_new, torch), bf16_dev(st.v_new, torch), kp, vp)
    return shape, runner, kp, vp, bf16_dev(st.q, torch)


def _call_static(lib, st, shape, runner, kp, vp, q, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.paged_attention_step_static_scratch(
        q.data_ptr(), kp.data_ptr(), vp.data_ptr(), runner.table.data_ptr(),
        int(runner.table.shape[1]), runner.cu.data_ptr(), runner.ctx.data_ptr(), st.B, st.T,
        runner.max_ctx, runner.items.data_ptr(), int(runner.items.numel() // bd.ITEM_INTS),
        out.data_ptr(), C.byref(shape), runner.err.data_ptr(), stream)


def test_static_scratch_matches_workspace_entry_point_twice(lib):
    steps = [wl.make_step(32, 8, 128, 16, [3000, 17, 1100, 2100], [1, 1, 77, 33], seed=41),
             wl.make_step(64, 8, 128, 32, [5000, 1025, 40], [1, 100, 1], seed=42)]
    for i, st in enumerate(steps):
        shape, runner, kp, vp, q = _prepare(st)
        assert bd.pa_workspace_bytes(shape, st.T, runner.max_ctx) <= STATIC_SCRATCH_BYTES
        ref_out = torch.empty((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        runner.attend(q, kp, vp, ref_out)
        out = torch.full((st.T, st.Hq, st.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call_static(lib, st, shape, runner, kp, vp, q, out) == bd.PA_OK
        torch.cuda.synchronize()
        if i > 0:
            # past the first call (which looks the array up on this device), a call takes
            # no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        assert runner.device_error() == 0
        got = out.view(torch.int16).cpu().numpy()
        want = ref_out.view(torch.int16).cpu().numpy()
        assert np.all(np.isfinite(pa.bf16_to_f64(got.view(np.uint16))))
        assert np.array_equal(got, want)
        # and, for the record, both are the oracle's attention within the parity tolerance
        d = np.abs(pa.bf16_to_f64(got.view(np.uint16)) -
                   pa.attention(st.q, kp.view(torch.int16).cpu().numpy().view(np.uint16),
                                vp.view(torch.int16).cpu().numpy().view(np.uint16),
                                st.block_table, st.cu_seqlens_q, st.ctx_lens, st.Hq))
        assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS


def test_static_scratch_refuses_steps_beyond_its_size(lib):
    # 2048 decode rows of 16k context need 2048 * 8 * 32 * 130 * 4 B of partials > 32 MiB
    st = wl.make_step(32, 8, 128, 16, [16384] * 2, [1, 1], seed=43, with_pool=False)
    shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    T = 2048
    assert bd.pa_workspace_bytes(shape, T, 16384) > STATIC_SCRATCH_BYTES
    p = dummy.data_ptr()
    st_code = lib.paged_attention_step_static_scratch(p, p, p, p, 1024, p, p, 2, T, 16384, p, 1,
                                                      p, C.byref(shape), None, None)
    assert st_code == bd.PA_ERR_WORKSPACE
