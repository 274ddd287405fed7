"""Pins for the oracle's NVFP4 operand format (no GPU): E2M1 codes in blocks of 16
with one E4M3 scale each.  Independent routes: hand-worked blocks
(tests/golden/nvfp4_blocks.txt), nearest-point brute force over the decoded E4M3
and E2M1 tables, special blocks, and scores recomputed from a decoder written
here from the bit layouts."""
import math
import os

import numpy as np
import pytest

import oracle
from workloads import to_bf16_bits, bf16_bits_to_f32

GOLD = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def e4m3_value(c):
    """E4M3 from its bits: bias 7, 3 mantissa bits, exponent field 0 subnormal."""
    e, m = (c >> 3) & 15, c & 7
    v = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if c & 0x80 else v


POS_E4M3 = [(c, e4m3_value(c)) for c in range(0x7F)]      # 0x7F is NaN


def nearest_even(cands, x):
    """(code, value) nearest to x; a tie goes to the even code."""
    best = min(abs(v - x) for _, v in cands)
    ties = [c for c, v in cands if abs(v - x) == best]
    return min(ties, key=lambda c: (c & 1, c))


def ref_block(xs):
    """NVFP4 of one block by exhaustive search (finite inputs)."""
    amax = max(abs(x) for x in xs)
    t = amax / 6
    sc = 0x7E if t >= 448 else nearest_even(POS_E4M3, t)
    s = e4m3_value(sc)
    codes = []
    for x in xs:
        if s == 0:
            codes.append(0)
            continue
        y = x / s
        mag = nearest_even(list(enumerate(E2M1)), min(abs(y), 6.0))
        codes.append(mag | (8 if math.copysign(1, y) < 0 else 0))
    return sc, codes


def test_hand_worked_blocks():
    for line in open(os.path.join(GOLD, "nvfp4_blocks.txt")):
        if line[0] == "#":
            continue
        name, vals, sc, codes = [f.strip() for f in line.split("|")]
        x = to_bf16_bits(np.array([[float(v) for v in vals.split()]], np.float32))
        c, s = oracle.nvfp4_quantize_rows(x)
        assert s[0, 0] == int(sc, 16), name
        assert list(c[0]) == [int(v) for v in codes.split()], name


@pytest.mark.parametrize("seed", range(4))
def test_matches_bruteforce_nearest(seed):
    rng = np.random.default_rng(seed)
    n = 400
    x = rng.standard_normal((n, 16)) * np.exp2(rng.integers(-14, 14, (n, 1)))
    x[::7, 3] = np.exp2(rng.integers(-8, 8, (n + 6) // 7)) * 0.75   # exact E2M1 ties at power-of-two scales
    xb = to_bf16_bits(x.astype(np.float32))
    xf = bf16_bits_to_f32(xb).astype(np.float64)
    c, s = oracle.nvfp4_quantize_rows(xb)
    for r in range(n):
        sc, codes = ref_block(list(xf[r]))
        assert s[r, 0] == sc, (r, xf[r])
        assert list(c[r]) == codes, (r, xf[r])


def test_special_blocks():
    z = np.zeros((4, 16), np.float32)
    z[1, 5] = np.inf
    z[2, :] = 1e-4                     # amax/6 below half the smallest E4M3 subnormal: scale 0
    z[3, :] = -3e5                     # saturation: scale 448, codes -6
    xb = to_bf16_bits(z)
    xb[1, 9] = 0x7FC0
    c, s = oracle.nvfp4_quantize_rows(xb)
    assert s[0, 0] == 0 and not c[0].any()
    assert s[1, 0] == 0x7F and not c[1].any()
    assert s[2, 0] == 0 and not c[2].any()
    assert s[3, 0] == 0x7E and (c[3] == 15).all()


def test_padding_and_block_index():
    x = np.concatenate([np.arange(1, 33), np.full(8, 0.5)]).astype(np.float32).reshape(1, 40)   # 2.5 blocks;
    # the partial block's small values make a padding of ones (instead of zeros) visible
    c, s = oracle.nvfp4_quantize_rows(to_bf16_bits(x))
    assert c.shape == (1, 48) and s.shape == (1, 3)
    assert not c[0, 40:].any()
    for b in range(3):
        sc, codes = ref_block(list(np.pad(x[0], (0, 8))[16 * b:16 * b + 16].astype(np.float64)))
        assert s[0, b] == sc and list(c[0, 16 * b:16 * b + 16]) == codes


def test_dequantisation_error_bound():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((300, 64)) * 3
    xb = to_bf16_bits(x.astype(np.float32))
    xf = bf16_bits_to_f32(xb).astype(np.float64)
    c, s = oracle.nvfp4_quantize_rows(xb)
    val = np.array([E2M1[v & 7] * (-1 if v & 8 else 1) for v in c.ravel()]).reshape(c.shape)
    sv = np.array([e4m3_value(int(v)) for v in s.ravel()]).reshape(s.shape)
    deq = val * np.repeat(sv, 16, axis=1)
    # within one E2M1 half-spacing (at most 1, between 4 and 6) of the scaled grid,
    # plus the scale's own rounding (the block max lands within 6 +- 1 of x/s)
    assert np.all(np.abs(deq - xf) <= np.repeat(sv, 16, axis=1) * 1.0 + 1e-12)


def test_scores_are_dot_products_of_decoded_operands():
    """fsa_emulate with NVFP4 Q/K: the raw scores are fp32 dot products of the
    operands decoded here from their bits (not through the oracle's decoder)."""
    rng = np.random.default_rng(3)
    B, H, S, D = 1, 2, 96, 128
    q, k, v = [to_bf16_bits(rng.standard_normal((B, H, S, D)).astype(np.float32)) for _ in range(3)]
    mx = oracle.MxInputs.from_bf16(q, k, v, 5, 0)
    res = oracle.fsa_emulate(mx, S, False, 0.125, 0, np.arange(B * H * S), dump=True)
    dec = lambda c, s: (np.array([E2M1[x & 7] * (-1 if x & 8 else 1) for x in c.ravel()]).reshape(c.shape) *
                        np.repeat(np.array([e4m3_value(int(x)) for x in s.ravel()]).reshape(s.shape), 16, axis=-1))
    qh, kh = dec(mx.qc, mx.qs), dec(mx.kc, mx.ks)
    for h in range(H):
        ref = (qh[0, h] @ kh[0, h].T).astype(np.float32)
        got = res["s"][h * S:(h + 1) * S, :S]
        assert np.array_equal(got, ref)
