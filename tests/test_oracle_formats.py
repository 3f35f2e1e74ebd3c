"""Pins for the oracle's number formats and NVFP4 quantiser (CPU only).

Each check ties the oracle to something outside itself: torch's own
float8_e4m3fn conversion, the E2M1 value set the OCP MX format defines, the
hand-worked groups in tests/golden/nvfp4_groups.txt, exact-rational brute force
and the bf16 representability claim of ROCm/ATOM #2745 (Validation).
"""
import itertools
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_groups.txt")


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e4m3_landmarks():
    assert formats.e4m3_value(0x38) == 1.0
    assert formats.e4m3_value(0x7E) == 448.0
    assert formats.e4m3_value(0x01) == 2.0 ** -9
    assert formats.e4m3_value(0x08) == 2.0 ** -6
    assert formats.e4m3_value(0xB8) == -1.0


def test_e2m1_values():
    # the E2M1 value set: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives
    assert formats.E2M1_TABLE[:8].tolist() == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert formats.E2M1_TABLE[8:].tolist() == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    assert np.signbit(formats.E2M1_TABLE[8])


def _f32_grid_and_midpoints(table, n):
    mags = sorted(set(abs(v) for v in table[:n].tolist()))
    pts = list(mags)
    pts += [(a + b) / 2 for a, b in zip(mags, mags[1:])]
    return pts


def test_e4m3_encode_matches_torch():
    rng = np.random.default_rng(7)
    mids = _f32_grid_and_midpoints(formats.E4M3_TABLE, 0x7F)
    x = np.concatenate([
        rng.standard_normal(20000) * 30,
        rng.uniform(-448, 448, 20000),
        rng.standard_normal(5000) * 1e-3,
        np.array(mids), -np.array(mids),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = formats.e4m3_encode(x)
    # torch maps -0 results to 0x80 like we do; compare bytes
    assert np.array_equal(ref, ours)


def test_e4m3_encode_saturates():
    x = np.array([448.0, 449.0, 464.0, 500.0, 1e9, -1e9], dtype=np.float32)
    assert formats.e4m3_encode(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def _e2m1_bruteforce(v: float) -> int:
    """Nearest E2M1 code by exact rational distance, ties to even mantissa,
    saturating at 6."""
    fv = Fraction(v)
    best = None
    for code in range(8):
        mag = Fraction(formats.e2m1_value(code))
        d = abs(abs(fv) - mag)
        key = (d, code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    code = best[1]
    if abs(fv) >= 6:
        code = 7
    if v < 0 or (v == 0 and np.signbit(v)):
        code |= 8
    return code


def test_e2m1_encode_bruteforce():
    rng = np.random.default_rng(11)
    mids = _f32_grid_and_midpoints(formats.E2M1_TABLE, 8)
    x = np.concatenate([rng.uniform(-8, 8, 4000), np.array(mids), -np.array(mids),
                        np.array([0.0, -0.0, 6.0, 7.0, -100.0, 1e-30, -1e-30])]).astype(np.float32)
    ours = formats.e2m1_encode(x)
    ref = np.array([_e2m1_bruteforce(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(ours, ref)


def _read_golden():
    cases = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals, sc, pay = [p.strip() for p in line.split("|")]
            x = [float(v) for v in vals.split()]
            assert len(x) == 16
            cases.append((x, int(sc, 16), [int(b, 16) for b in pay.split()]))
    return cases


def _bf16_bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", _read_golden())
def test_nvfp4_golden_groups(case):
    x, sc, pay = case
    key = np.zeros((1, 128), dtype=np.uint16)
    # place the group in every one of the 8 group slots of a key, in turn
    for g in range(8):
        key[:] = 0
        key[0, 16 * g:16 * g + 16] = _bf16_bits(x)
        payload, scale = formats.nvfp4_quantize(key)
        assert scale[0, g] == sc, (g, hex(scale[0, g]))
        assert payload[0, 8 * g:8 * g + 8].tolist() == pay, (g, payload[0].tolist())
        others = [h for h in range(8) if h != g]
        assert all(scale[0, h] == 0 for h in others)


def test_nvfp4_products_exact_in_bf16():
    """Every e2m1 x finite E4M3 product is a bf16 value (ROCm/ATOM #2745,
    Validation): this is why the FP4 scorer can equal a bf16 scorer fed the
    dequantised cache."""
    e2m1 = formats.E2M1_TABLE
    e4m3 = formats.E4M3_TABLE[~np.isnan(formats.E4M3_TABLE)]
    assert len(e4m3) == 254
    prod = np.array([a * b for a, b in itertools.product(e2m1, e4m3)], dtype=np.float64)
    back = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(prod, back)


def test_nvfp4_roundtrip_error_bound():
    """Dequantised values stay within one e2m1 half-step (1 x scale, the widest
    gap being 4..6) of an unsaturated input; a saturated input loses at most
    amax - 6 x scale, which is below amax/16 whenever the scale is a normal E4M3
    number (relative rounding <= 2^-4); a zero scale zeroes the group."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((512, 128)) * np.exp(rng.uniform(-6, 6, (512, 1)))).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xv = formats.bf16_bits_to_f32(bits).astype(np.float64)
    payload, scale = formats.nvfp4_quantize(bits)
    deq = formats.nvfp4_dequantize(payload, scale)
    s = np.repeat(formats.E4M3_TABLE[scale], 16, axis=1)
    amax = np.repeat(np.abs(xv).reshape(512, 8, 16).max(axis=2), 16, axis=1)
    err = np.abs(deq - xv)
    sat = np.abs(xv) > 6 * s
    assert np.all(err[~sat & (s > 0)] <= s[~sat & (s > 0)])
    assert np.all(err[sat & (s > 0)] <= (amax - 6 * s)[sat & (s > 0)])
    normal = s >= 2.0 ** -6
    assert np.all((amax - 6 * s)[normal] <= amax[normal] / 16)
    assert np.all(deq[s == 0] == 0)
    # signs never flip
    assert np.all(deq * xv >= 0)


def test_bf16_bits_roundtrip():
    v = torch.randn(1000, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bits = v.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(formats.bf16_bits_to_f32(bits), v.to(torch.float32).numpy())
