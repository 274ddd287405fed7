"""Pins for the oracle's scalar codecs and MX quantiser (no GPU).

Every check uses an independent route: format tables from the OCP MX standard
(tests/golden), exhaustive round trips, nearest-point brute force over the
decoded table, and hand-worked scale exponents."""
import math
import os

import numpy as np
import pytest

import oracle
from workloads import to_bf16_bits, bf16_bits_to_f32

GOLD = os.path.join(os.path.dirname(__file__), "golden")
NBITS = {0: 8, 1: 6, 2: 4, 4: 6}


def test_e2m1_table_matches_ocp():
    rows = [l.split() for l in open(os.path.join(GOLD, "e2m1_values.txt")) if l[0] != "#"]
    for code, val in rows:
        got = oracle.decode(2, int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_format_limits_match_ocp():
    for l in open(os.path.join(GOLD, "format_limits.txt")):
        if l[0] == "#":
            continue
        name, mx, mn, msub, emax, nans = l.split()
        f = oracle.FMT[name]
        n = NBITS[f]
        vals = [oracle.decode(f, c) for c in range(1 << n)]
        fin = [v for v in vals if not math.isnan(v)]
        assert max(fin) == float(mx)
        assert min(v for v in fin if v > 0) == float(msub)
        assert oracle.EMAX[f] == int(emax) == math.floor(math.log2(float(mx)))
        nan_codes = [c for c, v in enumerate(vals) if math.isnan(v)]
        assert nan_codes == ([] if nans == "none" else [int(x, 16) for x in nans.split(",")])
        # smallest normal: exponent field 1, mantissa 0
        mbits = {0: 3, 1: 3, 2: 1, 4: 2}[f]
        assert oracle.decode(f, 1 << mbits) == float(mn)


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_roundtrip_every_code(fmt):
    for c in range(1 << NBITS[fmt]):
        v = oracle.decode(fmt, c)
        if math.isnan(v):
            continue
        assert oracle.encode(fmt, v) == c, (fmt, c, v)


def _nearest_even_bruteforce(fmt, x):
    """Nearest decoded value by exhaustive search; ties to the even code."""
    n = NBITS[fmt]
    best = None
    for c in range(1 << n):
        v = oracle.decode(fmt, c)
        if math.isnan(v) or math.copysign(1, v) != math.copysign(1, x):
            continue
        d = abs(v - x)
        key = (d, c & 1)            # smaller distance, then even mantissa LSB
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_encode_matches_bruteforce_nearest(fmt):
    rng = np.random.default_rng(5)
    mx = oracle.decode(fmt, (1 << (NBITS[fmt] - 1)) - (2 if fmt == 0 else 1))
    xs = list(rng.uniform(-1.2 * mx, 1.2 * mx, 3000)) + list(rng.standard_normal(1000) * 0.3)
    # every midpoint between neighbouring grid values (the ties)
    pos = sorted({oracle.decode(fmt, c) for c in range(1 << (NBITS[fmt] - 1))} - {float("nan")})
    pos = [p for p in pos if not math.isnan(p)]
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    xs += mids + [-m for m in mids]
    for x in xs:
        x = float(x)
        if abs(x) >= mx:
            continue            # saturation checked separately
        assert oracle.encode(fmt, x) == _nearest_even_bruteforce(fmt, x), (fmt, x)


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_saturation_and_signed_zero(fmt):
    n = NBITS[fmt]
    sign = 1 << (n - 1)
    mx = max(v for v in (oracle.decode(fmt, c) for c in range(sign)) if not math.isnan(v))
    assert oracle.decode(fmt, oracle.encode(fmt, mx * 1.07)) == mx
    assert oracle.decode(fmt, oracle.encode(fmt, 1e30)) == mx
    assert oracle.decode(fmt, oracle.encode(fmt, -1e30)) == -mx
    assert oracle.encode(fmt, 0.0) == 0
    assert oracle.encode(fmt, -0.0) == sign
    tiny = oracle.decode(fmt, 1) / 4          # below half the smallest subnormal
    assert oracle.encode(fmt, -tiny) == sign
    assert oracle.encode(fmt, oracle.decode(fmt, 1) / 2) == 0    # exact tie to even zero


def test_e8m0():
    assert oracle.decode(3, 127) == 1.0
    assert oracle.decode(3, 0) == 2.0 ** -127
    assert oracle.decode(3, 254) == 2.0 ** 127
    assert math.isnan(oracle.decode(3, 255))


# --------------------------------------------------------------------------- MX quantiser
def _bf16(x):
    return to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("fmt,emax", [(0, 8), (1, 2), (2, 2), (4, 4)])
def test_mx_scale_hand_cases(fmt, emax):
    # amax = 1.0 -> floor(log2) = 0 -> E = -emax; amax = 3.0 -> 1 - emax; amax = 0.75 -> -1 - emax
    for amax, fl in [(1.0, 0), (3.0, 1), (0.75, -1), (2.0 ** -20, -20), (1000.0, 9)]:
        x = np.zeros((1, 32), np.float32)
        x[0, 5] = amax
        x[0, 6] = -amax / 3
        c, s = oracle.mx_quantize_rows(_bf16(x), fmt)
        assert s[0, 0] == 127 + fl - emax
    c, s = oracle.mx_quantize_rows(_bf16(np.zeros((1, 32))), fmt)
    assert s[0, 0] == 0 and not c.any()


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_mx_scale_clamps_at_minus_127(fmt):
    """E8M0 has no scale below 2^-127: a block whose max is 2^-126 (the smallest
    normal bf16) would want E = -126 - emax and gets -127 (scale byte 0); the max
    element then carries the factor 2^(127 - 126) = 2 in its code."""
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = 2.0 ** -126
    c, s = oracle.mx_quantize_rows(_bf16(x), fmt)
    assert s[0, 0] == 0
    assert oracle.decode(fmt, int(c[0, 5])) == 2.0


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_mx_exact_roundtrip_on_representable(fmt):
    """x = decode(code) * 2^E with the block max at the format's top binade
    quantises back to the same codes and the scale byte E + 127."""
    rng = np.random.default_rng(11)
    n = NBITS[fmt]
    sign = 1 << (n - 1)
    codes = [c for c in range(1 << n) if not math.isnan(oracle.decode(fmt, c))]
    emax = oracle.EMAX[fmt]
    top = [c for c in range(sign) if not math.isnan(oracle.decode(fmt, c))
           and 2.0 ** emax <= oracle.decode(fmt, c)]
    for trial in range(50):
        E = int(rng.integers(-100, 100))
        cc = rng.choice(codes, 32)
        cc[rng.integers(32)] = rng.choice(top)
        x = np.array([oracle.decode(fmt, int(c)) * 2.0 ** E for c in cc], np.float64)
        xb = _bf16(x.astype(np.float32))
        assert np.array_equal(bf16_bits_to_f32(xb).astype(np.float64), x)   # bf16-exact
        c, s = oracle.mx_quantize_rows(xb[None, :], fmt)
        assert s[0, 0] == E + 127
        dec = np.array([oracle.decode(fmt, int(k)) for k in c[0]])
        assert np.array_equal(dec * 2.0 ** E, x)


def test_mx_error_bound_and_padding():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((7, 50)).astype(np.float32) * 5)
    for fmt, mbits in [(0, 3), (1, 3), (2, 1), (4, 2)]:
        c, s = oracle.mx_quantize_rows(x, fmt)
        assert c.shape == (7, 64) and s.shape == (7, 2)
        assert not c[:, 50:].any()                                       # zero padding
        xf = bf16_bits_to_f32(x).astype(np.float64)
        E = s.astype(np.int64) - 127
        dec = oracle.decode_array(fmt, c)[:, :50] * 2.0 ** np.repeat(E, 32, axis=1)[:, :50]
        # error <= half a grid step at the block's top binade (or saturation at 2^(emax+1))
        Ee = np.repeat(E, 32, axis=1)[:, :50]
        step = 2.0 ** (Ee + oracle.EMAX[fmt] - mbits)
        top = {0: 448.0, 1: 7.5, 2: 6.0, 4: 28.0}[fmt] * 2.0 ** Ee
        inside = np.abs(xf) <= top
        assert np.all(np.abs(dec - xf)[inside] <= step[inside] * 0.5)
        assert np.array_equal(dec[~inside], np.sign(xf[~inside]) * top[~inside])   # satfinite


def test_mx_cols_blocks_along_sequence():
    rng = np.random.default_rng(4)
    v = _bf16(rng.standard_normal((1, 2, 70, 64)).astype(np.float32))
    c, s = oracle.mx_quantize_cols(v, 0)
    assert c.shape == (1, 2, 64, 96) and s.shape == (1, 2, 64, 3)
    c2, s2 = oracle.mx_quantize_rows(np.ascontiguousarray(np.swapaxes(v, 2, 3)), 0)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


@pytest.mark.parametrize("fmt", [0, 1, 2, 4])
def test_mx_nonfinite_block(fmt):
    """A block with an Inf takes the E8M0 NaN scale 0xFF (OCP MX: the whole block
    then decodes to NaN).  Its element codes: the E4M3 NaN code 0x7F, or 0 in the
    formats that have no NaN encoding; the finite neighbour block is untouched."""
    x = np.ones((1, 64), np.float32)
    x[0, 40] = np.inf
    c, s = oracle.mx_quantize_rows(_bf16(x), fmt)
    assert s[0, 1] == 0xFF and s[0, 0] == 127 - oracle.EMAX[fmt]
    assert np.all(c[0, 32:] == (0x7F if fmt == 0 else 0))
    assert math.isnan(oracle.decode(3, int(s[0, 1])))


def test_encode_nan_keeps_sign_e4m3():
    """E4M3 encodes NaN as S.1111.111 (OCP); the encoder keeps the sign of the NaN."""
    assert oracle.encode(0, float("nan")) == 0x7F
    assert oracle.encode(0, -float("nan")) == 0xFF
    assert math.isnan(oracle.decode(0, 0x7F)) and math.isnan(oracle.decode(0, 0xFF))
