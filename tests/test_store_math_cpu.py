"""The NVFP4 store's division-free code rule, checked exhaustively on the CPU.

The store kernel quantises a bf16 value v with an E4M3 scale s to the e2m1 code
of q = fl(v / s) (ATOM #2745, Summary, "Store": codes of x / scale, rounded
half-to-even, saturating at 6) without a correctly rounded division.  Its
argument: each product t * s of an e2m1 midpoint t and a scale is exact and
itself a bf16 value, so a bf16 v is either exactly at t * s or a bf16 spacing
away from it, and the rounding of the quotient can never carry it across t.
This test checks the consequence, that comparing |v| with t * s decides every
midpoint comparison of fl(v / s), for every finite bf16 magnitude against every
positive finite E4M3 scale, with numpy's IEEE fp32 division as the reference.
"""
import numpy as np

# the e2m1 grid's midpoints and whether the quotient must exceed or reach them
# (ties go to the code whose mantissa bit is zero)
MIDPOINTS = [(0.25, ">"), (0.75, ">="), (1.25, ">"), (1.75, ">="), (2.5, ">"), (3.5, ">="),
             (5.0, ">")]


def _e4m3(code: int) -> np.float32:
    e, m = (code >> 3) & 15, code & 7
    return np.float32(m * 2.0 ** -9) if e == 0 else np.float32((8 + m) * 2.0 ** (e - 10))


def test_scaled_midpoints_give_the_codes_of_the_rounded_quotient():
    v = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)  # all finite bf16 >= 0
    mismatches = 0
    with np.errstate(over="ignore"):
        for code in range(1, 127):                  # 0 is zero, 0x7f is NaN
            s = _e4m3(code)
            q = (v / s).astype(np.float32)          # correctly rounded fp32 quotient
            by_quotient = np.zeros(v.shape, np.int32)
            by_product = np.zeros(v.shape, np.int32)
            for t, op in MIDPOINTS:
                ts = np.float32(t) * s
                assert float(ts) == t * float(s), "t * s must be exact in fp32"
                assert int(ts.view(np.uint32)) & 0xFFFF == 0, "t * s must be a bf16 value"
                if op == ">":
                    by_quotient += q > np.float32(t)
                    by_product += v > ts
                else:
                    by_quotient += q >= np.float32(t)
                    by_product += v >= ts
            mismatches += int(np.count_nonzero(by_quotient != by_product))
    assert mismatches == 0


def test_a_planted_off_by_one_product_is_caught():
    # the same check with one midpoint's comparison flipped must fail somewhere
    v = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    s = _e4m3(0x38)  # 1.0
    q = (v / s).astype(np.float32)
    assert np.count_nonzero((q > np.float32(0.75)) != (v >= np.float32(0.75) * s)) > 0
