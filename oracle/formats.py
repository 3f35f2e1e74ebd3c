"""Number formats of the index-K cache, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* E4M3 (OCP 8-bit floating point, "fn" variant): 1 sign bit, 4 exponent bits
  with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
  m/8 * 2^-6; S.1111.111 is NaN; there are no infinities; largest finite 448.
* E2M1 (OCP MX 4-bit floating point): 1 sign bit, 2 exponent bits with bias 1,
  1 mantissa bit; exponent field 0 encodes 0 and 0.5; largest value 6; no
  infinities or NaN.
* NVFP4 index key as ROCm/ATOM #2745 describes it (Summary, per cached key with
  D = 128): a 64-byte e2m1 payload, two codes per byte with the even element in
  the low nibble, plus 8 bytes of E4M3 block scales, one per 16 elements, with a
  unit outer scale.  The store quantises each group of 16 with
  scale = e4m3(amax / 6) and codes rounded half-to-even that saturate at 6.

Readings where the page is silent (each listed in the design notes):
  amax and amax/6 are fp32; amax/6 is rounded to E4M3 half-to-even and
  saturated at 448; a scale that rounds to 0 makes the whole group's codes 0;
  each code is e2m1(x / s) with x / s a correctly rounded fp32 division; the
  sign of a negative value that rounds to zero is kept (code 0x8).
"""
from __future__ import annotations

import numpy as np

E4M3_SIGN = 0x80
E2M1_SIGN = 0x8
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def e4m3_value(code: int) -> float:
    """Value of one E4M3 byte (NaN for the two NaN encodings)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e2m1_value(code: int) -> float:
    """Value of one E2M1 nibble."""
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return sign * (m / 2.0)
    return sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def _encode_rne_sat(x: np.ndarray, magnitudes: np.ndarray, sign_bit: int) -> np.ndarray:
    """Round each value to the nearest grid point, ties to the even code
    (mantissa LSB 0), magnitudes beyond the largest saturate to it.

    ``magnitudes[c]`` is the value of non-negative code ``c``; it rises with c,
    so the code of a grid point is its index and its mantissa LSB is bit 0.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = len(magnitudes) - 1
    lo = np.clip(np.searchsorted(magnitudes, a, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    d_lo = a - magnitudes[lo]
    d_hi = magnitudes[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= magnitudes[top], top, code)          # saturate
    code = np.where(np.signbit(x), code | sign_bit, code)     # sign kept, -0 included
    return code.astype(np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 round-to-nearest-even, saturating at 448 (finite inputs)."""
    mags = E4M3_TABLE[:0x7F]             # codes 0x00..0x7E (0x7F is NaN)
    return _encode_rne_sat(x, mags, E4M3_SIGN)


def e2m1_encode(x) -> np.ndarray:
    """E2M1 round-to-nearest-even, saturating at 6 (finite inputs)."""
    mags = E2M1_TABLE[:8]
    return _encode_rne_sat(x, mags, E2M1_SIGN)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> their exact float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def nvfp4_quantize(keys_bf16_bits: np.ndarray):
    """Quantise keys [T, 128] (bf16 bit patterns) to NVFP4 planes.

    Follows ROCm/ATOM #2745, Summary: per group of 16 elements,
    scale = e4m3(amax / 6); codes = e2m1(x / scale), half-to-even, saturating
    at 6; payload byte b holds element 2b in its low nibble, 2b+1 in its high.
    Returns (payload uint8 [T, 64], scale uint8 [T, 8]).
    """
    x = bf16_bits_to_f32(keys_bf16_bits)
    T, D = x.shape
    assert D % 16 == 0
    g = x.reshape(T, D // 16, 16)
    amax = np.abs(g).max(axis=2).astype(np.float32)
    s_f = (amax / np.float32(6.0)).astype(np.float32)            # fp32 division
    s_code = e4m3_encode(s_f)
    s_val = E4M3_TABLE[s_code].astype(np.float32)                # exact in fp32
    safe = np.where(s_val > 0, s_val, np.float32(1.0)).astype(np.float32)
    v = (g / safe[:, :, None]).astype(np.float32)                # fp32 division
    codes = e2m1_encode(v).reshape(T, D // 16, 16)
    codes = np.where((s_val > 0)[:, :, None], codes, 0).astype(np.uint8)
    codes = codes.reshape(T, D)
    payload = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return payload, s_code.astype(np.uint8)


def nvfp4_dequantize(payload: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """NVFP4 planes [T, 64] + [T, 8] -> float64 keys [T, 128]:
    e2m1(nibble) x e4m3(scale of its group of 16), unit outer scale."""
    p = np.asarray(payload, dtype=np.uint8)
    T = p.shape[0]
    codes = np.empty((T, p.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    vals = E2M1_TABLE[codes]
    sc = E4M3_TABLE[np.asarray(scale, dtype=np.uint8)]
    return vals * np.repeat(sc, 16, axis=1)


def fp8_dequantize(codes: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """E4M3 keys [T, 128] with one little-endian fp32 scale per key (scale
    plane rows of 4 bytes) -> float64 code value x scale."""
    s = np.ascontiguousarray(scale_bytes, dtype=np.uint8).view("<f4").reshape(-1)
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)] * s.astype(np.float64)[:, None]


def bf16_dequantize(payload: np.ndarray) -> np.ndarray:
    """bf16 keys stored as 256-byte little-endian rows -> float64 [T, 128]."""
    bits = np.ascontiguousarray(payload, dtype=np.uint8).view("<u2")
    return bf16_bits_to_f32(bits).astype(np.float64)
