"""FP8 (float8_e4m3fn) KV cache with per-tensor scales, as plain definitions.

Test infrastructure only (see the package docstring): the product never imports this.

What the pages fix:
  [P3-review] "P3: native paged-KV continuous-batching sampler", Review (the kv_dtype item):
      K/V are dequantised on read; float8_e4m3fn used UNSCALED is visibly lossy, so an fp8
      KV cache needs per-tensor scales, not just a dtype switch.
  [P3-tp]     same page, Tensor parallelism, open item 6: fp8 KV with per-tensor scales.
  [RL-4.2]    "Finish RL Training Faster: Bitwise-Consistent, High-Performance, Agent-Driven",
      section 4.2: keep FP8 storage, one read path for prefill and decode, one shared write
      path; section 4.4 item 1: quantisation rounds to nearest, element by element.

The format (float8_e4m3fn): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
Exponent field 0 holds the subnormals m/8 * 2^-6; fields 1..15 hold (1 + m/8) * 2^(e-7);
field 15 with mantissa 7 is NaN (either sign); there are no infinities, so the largest
finite value is (1 + 6/8) * 2^8 = 448.

Readings where the pages leave a step open (each also listed in the design notes):
  F1  One scale per tensor: s_k for every K element of the pool, s_v for every V element.
      The caller chooses them (for example amax / 448 of what it will write).
  F2  Write: code = e4m3(x / s), with x the bf16 value widened to fp32, the division in
      fp32 (IEEE round to nearest), then rounding to the nearest e4m3 value, ties to the
      even code, and saturation of finite values beyond 448 to +-448 (no NaN from a finite
      input). A NaN input gives the NaN code.
  F3  Read: the dequantised value is code_value * s, taken exactly (fp64 here).
"""
from __future__ import annotations

import numpy as np

__all__ = ["E4M3_MAX", "decode_e4m3", "encode_e4m3", "quantize", "dequantize",
           "e4m3_values"]

E4M3_MAX = 448.0
_NAN_CODE = 0x7F


def e4m3_values() -> np.ndarray:
    """fp64 value of each of the 256 codes, straight from the format definition."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_VALUES = e4m3_values()
_POS = _VALUES[:0x7F]          # codes 0x00 .. 0x7E: the non-negative finite values, ascending


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """fp64 values of uint8 codes (exact)."""
    return _VALUES[np.asarray(codes, dtype=np.uint8)]


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """uint8 codes of float values: nearest e4m3 value, ties to the even code, finite values
    beyond 448 saturate to +-448, NaN gives the NaN code (F2)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # the neighbours lo <= a <= hi among the non-negative finite values
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, len(_POS) - 1)
    lo = np.clip(hi - 1, 0, None)
    d_lo = np.abs(a - _POS[lo])
    d_hi = np.abs(_POS[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a >= E4M3_MAX, np.uint8(0x7E), code)          # saturate
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(_NAN_CODE), code).astype(np.uint8)


def _quantize_values(x_bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    bits = np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    x32 = bits.view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        q32 = x32 / np.float32(scale)                     # fp32 division, round to nearest
    return encode_e4m3(q32.astype(np.float64))


def quantize(x_bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """KV-write codes of bf16 values (uint16 bit patterns) under one per-tensor scale (F2).

    A bf16 input has 65,536 possible bit patterns, so the definition is evaluated once for
    each of them and the codes are looked up: the same result as evaluating it per element,
    at a cost independent of the pool size."""
    table = _quantize_values(np.arange(65536, dtype=np.uint32).astype(np.uint16), scale)
    return table[np.asarray(x_bf16_bits, dtype=np.uint16)]


def dequantize(codes: np.ndarray, scale: float) -> np.ndarray:
    """The value a read of the cache stands for: code_value * scale, exactly (F3)."""
    return decode_e4m3(codes) * float(np.float32(scale))
