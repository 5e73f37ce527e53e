"""Pins for the float8_e4m3fn KV-cache oracle (oracle/fp8.py) against what the format and
the mathematics fix, and against an independent library cast (torch.float8_e4m3fn).
Pages: "P3: native paged-KV continuous-batching sampler", Review (kv_dtype item: dequantise
on read, per-tensor scales); "Finish RL Training Faster: Bitwise-Consistent, ...", 4.2
(FP8 storage, shared write path) and 4.4 item 1 (round to nearest, element by element)."""
import numpy as np
import pytest

from oracle import fp8
import oracle.paged_attention as pa


def test_format_fixed_points():
    v = fp8.e4m3_values()
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0          # largest finite value
    assert v[0x08] == 2.0 ** -6                             # smallest normal
    assert v[0x01] == 2.0 ** -9                             # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9                         # largest subnormal
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert v[0x40] == 2.0 and v[0x3C] == 1.5
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(v).sum() == 254
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                         # codes order the values


def test_decode_matches_torch_for_all_codes():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.decode_e4m3(codes)
    both_nan = np.isnan(t) & np.isnan(ours)
    assert np.all(both_nan | (t == ours))
    assert np.array_equal(np.signbit(t[~np.isnan(t)]), np.signbit(ours[~np.isnan(ours)]))


def test_encode_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 60, 20000),
                        rng.uniform(-440, 440, 20000), rng.normal(0, 0.01, 20000)])
    x = x.astype(np.float32).astype(np.float64)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode_e4m3(x), t)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.encode_e4m3(fp8.decode_e4m3(codes)), codes)


def test_ties_go_to_the_even_code_and_nearest_otherwise():
    pos = fp8.e4m3_values()[:0x7F]
    mid = (pos[:-1] + pos[1:]) / 2                          # exact in fp64
    got = fp8.encode_e4m3(mid)
    lo = np.arange(len(mid))
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got.astype(np.int64), want)
    # just off the midpoint the nearest value wins
    assert np.array_equal(fp8.encode_e4m3(np.nextafter(mid, -np.inf)).astype(np.int64), lo)
    assert np.array_equal(fp8.encode_e4m3(np.nextafter(mid, np.inf)).astype(np.int64), lo + 1)


def test_saturation_signs_and_nan():
    got = fp8.encode_e4m3(np.array([448.0, 463.9, 464.0, 1e6, np.inf, -1e6, -np.inf,
                                    np.nan, -0.0, -1e-12]))
    assert list(got[:7]) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert got[7] == 0x7F and got[8] == 0x80 and got[9] == 0x80


def test_quantisation_error_bound_and_scale():
    rng = np.random.default_rng(12)
    x = rng.normal(0, 3, 50000).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)      # truncation is fine for inputs
    xs = pa.bf16_to_f64(bits)
    s = float(np.float32(np.abs(xs).max() / 448.0))
    codes = fp8.quantize(bits, s)
    back = fp8.dequantize(codes, s)
    # round to nearest: error at most half a step, 2^-4 of the value for normals, and half
    # the subnormal step 2^-10 * s below the normal range
    err = np.abs(back - xs)
    bound = np.maximum(np.abs(xs) * 2.0 ** -4, 2.0 ** -10 * s)
    assert np.all(err <= bound * (1 + 1e-12))
    # the scale matters for small values: unscaled, data of magnitude ~1e-3 falls into the
    # e4m3 subnormals (step 2^-9) and loses most of its precision; scaled it keeps 2^-4
    small = (rng.normal(0, 1e-3, 20000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    xs2 = pa.bf16_to_f64(small)
    s2 = float(np.float32(np.abs(xs2).max() / 448.0))
    rel = lambda b: np.median(np.abs(b - xs2) / np.maximum(np.abs(xs2), 1e-30))
    assert rel(fp8.dequantize(fp8.quantize(small, s2), s2)) < 2.0 ** -5
    assert rel(fp8.dequantize(fp8.quantize(small, 1.0), 1.0)) > 2.0 ** -3


def test_quantize_divides_in_fp32():
    # 1/3 is not exact in fp32: x / s rounds once before the e4m3 rounding
    bits = np.array([0x3F80], dtype=np.uint16)              # 1.0
    s = 3.0
    q32 = np.float32(1.0) / np.float32(s)
    assert fp8.quantize(bits, s)[0] == fp8.encode_e4m3(np.array([float(q32)]))[0]


def test_mutant_truncating_quantiser_is_caught():
    """Rounding toward zero instead of to nearest must fail the nearest / tie pins."""
    def truncating(x):
        pos = fp8.e4m3_values()[:0x7F]
        a = np.abs(np.asarray(x, dtype=np.float64))
        idx = np.clip(np.searchsorted(pos, a, side="right") - 1, 0, 0x7E)
        return idx.astype(np.uint8)
    pos = fp8.e4m3_values()[:0x7F]
    just_above_mid = np.nextafter((pos[:-1] + pos[1:]) / 2, np.inf)
    assert not np.array_equal(truncating(just_above_mid), fp8.encode_e4m3(just_above_mid))


def test_dequantised_attention_reduces_to_the_bf16_oracle_on_exact_values():
    """With a power-of-two scale every dequantised value is exactly a bf16 value, so the
    attention over codes + scale equals the plain oracle over a bf16 pool holding those
    values: dequantisation is a storage change only."""
    rng = np.random.default_rng(13)
    s = 0.25
    shape = (4, 16, 2, 64)
    codes_k = (rng.integers(0, 0x7E, size=shape) | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)
    codes_v = (rng.integers(0, 0x7E, size=shape) | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)
    kf = fp8.dequantize(codes_k, s)
    vf = fp8.dequantize(codes_v, s)
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kb, vb = to_bf16(kf), to_bf16(vf)
    assert np.array_equal(pa.bf16_to_f64(kb), kf) and np.array_equal(pa.bf16_to_f64(vb), vf)
    q = to_bf16(rng.normal(0, 0.05, size=(3, 4, 64)))
    table = np.array([[2, 0, 3, 1]], dtype=np.int32)
    cu = np.array([0, 3], dtype=np.int32)
    ctx = np.array([50], dtype=np.int32)
    got = pa.attention(q, kf, vf, table, cu, ctx, 4)
    want = pa.attention(q, kb, vb, table, cu, ctx, 4)
    assert np.array_equal(got, want)


def test_table_quantiser_equals_the_per_element_definition():
    rng = np.random.default_rng(14)
    bits = rng.integers(0, 65536, size=200000).astype(np.uint16)
    for s in (0.011, 1.0, 3.0, 1e-30, 7e30):
        assert np.array_equal(fp8.quantize(bits, s), fp8._quantize_values(bits, s))
