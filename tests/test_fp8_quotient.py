"""The FP8 append's division-free quotient (CPU).

The append kernels store the E4M3 code of the correctly rounded float32
quotient x / s.  They compute it without a division: q0 = RN(x * r) with
r = RN(1 / s), then one fused multiply-add correction, q = RN(q0 + e * r) with
e = x - s * q0 exact (Markstein's final division step), taken only where the
last ulp can change the code (2^-11 <= |q0| <= 512).  This test restates that
arithmetic in numpy, with the fused multiply-adds emulated exactly, and checks
that it gives the oracle's code of the IEEE quotient for every bf16 input at
a few hundred scales, adversarial ones included (significands of all ones,
powers of two, scales far from 1)."""
import numpy as np


def _rn32_sum(a, b):
    # RN32(a + b) for float64 a, b: the float64 sum and its exact two-sum error
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)
    f = s.astype(np.float32)
    f64 = f.astype(np.float64)
    up = np.nextafter(f, np.float32(np.inf))
    dn = np.nextafter(f, np.float32(-np.inf))
    at_up = s == (f64 + up.astype(np.float64)) / 2
    at_dn = s == (f64 + dn.astype(np.float64)) / 2
    res = np.where(at_up & (err > 0), up, f)
    return np.where(at_dn & (err < 0), dn, res)


def _codes_division_free(orc, x, s):
    y = np.float32(1.0) / s
    with np.errstate(all="ignore"):
        q0 = x * y
        e = (x.astype(np.float64) - np.float64(s) * q0.astype(np.float64)).astype(np.float32)
        q1 = _rn32_sum(q0.astype(np.float64), e.astype(np.float64) * np.float64(y))
    a = np.abs(q0)
    q = np.where((a >= np.float32(2.0 ** -11)) & (a <= np.float32(512.0)), q1, q0)
    return orc.e4m3_encode(q)


def test_division_free_codes_equal_ieee_quotient_codes(orc):
    bits = np.arange(0, 0x10000, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(11)
    scales = [0.0123, 0.0171, 0.25, 1.0 / (1.0625 * (1 + 3 * 2.0 ** -24)), 1.0, 3.0, 0.1, 7.0, 1e-3,
              2 - 2 ** -23, 1 + 2 ** -23, 1.5 - 2 ** -23, 2.0 ** -40, 2.0 ** 40, 1e-12, 1e12]
    scales += list(np.exp(rng.uniform(np.log(1e-4), np.log(1e4), 150)))
    scales += list(rng.integers(1 << 23, 1 << 24, 50) * 2.0 ** -23)
    for s in scales:
        s = np.float32(s)
        with np.errstate(all="ignore"):
            ref = orc.e4m3_encode(x / s)
        got = _codes_division_free(orc, x, s)
        assert np.array_equal(got, ref), (float(s), int(np.sum(got != ref)))


def test_a_plain_product_is_not_enough(orc):
    # x = 3 at scale 11.294117 (3/s = 0.265625 (1 + ~2^-24), just above the
    # midpoint 0.265625 between the E4M3 values 0.25 and 0.28125): the float32
    # quotient rounds up, the plain product x * RN(1/s) lands on the midpoint
    # and rounds to even; the correction step restores the quotient's code
    x = np.array([3.0], np.float32)
    s = np.float32(11.294116973876953)
    with np.errstate(all="ignore"):
        naive = orc.e4m3_encode(x * (np.float32(1.0) / s))
        ref = orc.e4m3_encode(x / s)
    assert naive[0] != ref[0]
    assert np.array_equal(_codes_division_free(orc, x, s), ref)
