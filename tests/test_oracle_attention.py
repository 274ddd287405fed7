"""Pins for the oracle's attention functions (no GPU): closed forms, invariants
and special cases that reduce to textbook results."""
import math

import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, Workload, bf16_bits_to_f32, generate, sample_rows, small, to_bf16_bits


def bf(x):
    return to_bf16_bits(np.asarray(x, np.float32))


def rnd(shape, seed, scale=1.0, integer=False):
    rng = np.random.default_rng(seed)
    if integer:
        return bf(rng.integers(-3, 4, shape).astype(np.float32))
    return bf(rng.standard_normal(shape).astype(np.float32) * scale)


def allrows(B, H, S):
    return np.arange(B * H * S, dtype=np.int64)


# --------------------------------------------------------------------------- exact attention
def test_exact_zero_query_gives_visible_mean():
    B, H, S, D = 1, 2, 40, 64
    q = bf(np.zeros((B, H, S, D)))
    k = rnd((B, H, S, D), 1)
    v = rnd((B, H, S, D), 2)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    for causal in (False, True):
        out = oracle.attn_exact(q, k, v, causal, 0.125, allrows(B, H, S))
        for h in range(H):
            for i in range(S):
                n = i + 1 if causal else S
                ref = vf[0, h, :n].mean(axis=0)
                assert np.allclose(out[h * S + i], ref, rtol=0, atol=1e-12)


def test_exact_two_keys_logistic():
    rng = np.random.default_rng(7)
    q = rnd((1, 1, 1, 64), 3)
    k = rnd((1, 1, 2, 64), 4)
    v = rnd((1, 1, 2, 64), 5)
    qf, kf, vf = (bf16_bits_to_f32(a).astype(np.float64) for a in (q, k, v))
    s = 0.125 * (kf[0, 0] @ qf[0, 0, 0])
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    out = oracle.attn_exact(q, k, v, False, 0.125, [0])[0]
    assert np.allclose(out, w0 * vf[0, 0, 0] + (1 - w0) * vf[0, 0, 1], atol=1e-13)


def test_exact_causal_row0_and_constant_v_and_shift_invariance():
    B, H, S, D = 1, 1, 33, 64
    q, k, v = rnd((B, H, S, D), 1, integer=True), rnd((B, H, S, D), 2, integer=True), rnd((B, H, S, D), 3)
    out = oracle.attn_exact(q, k, v, True, 0.125, allrows(B, H, S))
    assert np.array_equal(out[0], bf16_bits_to_f32(v)[0, 0, 0].astype(np.float64))
    ones = bf(np.ones((B, H, S, D)))
    assert np.allclose(oracle.attn_exact(q, k, ones, False, 0.125, allrows(B, H, S)), 1.0, atol=1e-14)
    # adding the same vector u to every key shifts a row's scores by q.u: softmax unchanged
    u = np.random.default_rng(9).integers(-2, 3, D).astype(np.float32)
    k2 = bf(bf16_bits_to_f32(k) + u)
    out2 = oracle.attn_exact(q, k2, v, True, 0.125, allrows(B, H, S))
    assert np.allclose(out, out2, atol=1e-12)


def test_exact_gqa_mapping():
    B, H, Hkv, S, D = 2, 4, 2, 20, 64
    q, k, v = rnd((B, H, S, D), 1), rnd((B, Hkv, S, D), 2), rnd((B, Hkv, S, D), 3)
    rows = allrows(B, H, S)
    out = oracle.attn_exact(q, k, v, False, 0.125, rows)
    k4, v4 = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    assert np.array_equal(out, oracle.attn_exact(q, k4, v4, False, 0.125, rows))


def test_exact_causal_rectangular_offset():
    # Sq < Sk: query i sees keys j <= i + Sk - Sq (bottom-right aligned)
    q, k, v = rnd((1, 1, 4, 64), 1), rnd((1, 1, 10, 64), 2), rnd((1, 1, 10, 64), 3)
    full = oracle.attn_exact(q, k[:, :, :7], v[:, :, :7], False, 0.125, [0])
    causal = oracle.attn_exact(q, k, v, True, 0.125, [0])
    assert np.allclose(full, causal, atol=1e-14)


# --------------------------------------------------------------------------- error floor
def test_floor_unquantised_p_equals_exact_on_representable_inputs():
    # integer inputs in [-3, 3] are exact in every MX format used here
    B, H, S, D = 1, 1, 70, 64
    q, k, v = (rnd((B, H, S, D), s, integer=True) for s in (1, 2, 3))
    for fq, fv in [(0, 0), (1, 1), (2, 2)]:
        mx = oracle.MxInputs.from_bf16(q, k, v, fq, fv)
        rows = allrows(B, H, S)
        fl = oracle.attn_floor(mx, S, True, 0.125, fv, rows, quantize_p=False)
        ex = oracle.attn_exact(q, k, v, True, 0.125, rows)
        assert np.allclose(fl, ex, atol=1e-12)


def test_floor_uniform_rows_and_error_order():
    B, H, S, D = 1, 1, 100, 64
    q0 = bf(np.zeros((B, H, S, D)))
    k, v = rnd((B, H, S, D), 2), rnd((B, H, S, D), 3)
    mx = oracle.MxInputs.from_bf16(q0, k, v, 0, 0)
    vh = oracle.decode_array(0, mx.vc) * 2.0 ** (np.repeat(mx.vs.astype(np.int64), 32, -1) - 127)
    out = oracle.attn_floor(mx, S, False, 0.125, 0, [0])
    assert np.allclose(out[0], vh[0, 0, :, :S].mean(axis=1), atol=1e-12)
    # quantising P adds error of the order of the P format's precision
    q = rnd((B, H, S, D), 1, 2.0)
    mx = oracle.MxInputs.from_bf16(q, k, v, 0, 0)
    rows = allrows(B, H, S)
    a = oracle.attn_floor(mx, S, False, 0.125, 0, rows, quantize_p=False)
    errs = []
    for fp, bound in [(0, 0.04), (1, 0.09), (2, 0.3)]:
        b = oracle.attn_floor(mx, S, False, 0.125, fp, rows, quantize_p=True)
        rel = np.linalg.norm(a - b) / np.linalg.norm(a)
        assert 0 < rel < bound, (fp, rel)
        errs.append(rel)
    assert errs[0] < errs[1] < errs[2]        # 3, 3 and 1 mantissa bits, narrower range for E2M3


def test_floor_and_emulate_use_each_blocks_own_scale():
    """Q and K rows whose two 32-element blocks differ in magnitude by 2^6 (every
    value exact in all three formats): with unquantised P the floor equals exact
    attention, which only holds if each block is dequantised with its own scale."""
    B, H, S, D = 1, 1, 70, 64
    rng = np.random.default_rng(8)
    def mixed(seed):
        x = np.random.default_rng(seed).integers(-3, 4, (B, H, S, D)).astype(np.float32)
        x[..., 32:] /= 64.0
        return bf(x)
    q, k, v = mixed(1), mixed(2), rnd((B, H, S, D), 3, integer=True)
    rows = allrows(B, H, S)
    ex = oracle.attn_exact(q, k, v, True, 0.5, rows)
    for fq in (0, 1, 2):
        mx = oracle.MxInputs.from_bf16(q, k, v, fq, fq)
        assert not np.array_equal(mx.qs[..., 0], mx.qs[..., 1])
        fl = oracle.attn_floor(mx, S, True, 0.5, fq, rows, quantize_p=False)
        assert np.allclose(fl, ex, atol=1e-12), fq


def test_floor_p_quantisation_closed_forms():
    """Closed forms of the floor's P quantisation (MX rule on 32-key blocks, E2M1 P).
    (a) Keys 0..15 score 0 and keys 16..31 score -4 share one block whose scale
        comes from p = 1 (E = 0 - 2): e^-4 * 2^2 = 0.073 rounds to code 0, so O is
        the mean of v over keys 0..15.
    (b) Two keys scoring 0 and -0.875: e^-0.875 * 2^2 = 1.667 rounds to 1.5, so
        p~ = (1, 0.375) and O = (v0 + 0.375 v1) / 1.375."""
    D = 64
    # (a) one query, q = e_0; k_j = (0 or -4) e_0; scale 1
    q = np.zeros((1, 1, 1, D), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, 32, D), np.float32)
    k[0, 0, 16:, 0] = -4.0
    v = np.random.default_rng(4).integers(-3, 4, (1, 1, 32, D)).astype(np.float32)
    mx = oracle.MxInputs.from_bf16(bf(q), bf(k), bf(v), 0, 2)
    out = oracle.attn_floor(mx, 32, False, 1.0, 2, [0])
    assert np.allclose(out[0], v[0, 0, :16].mean(axis=0), atol=1e-12)
    # (b) two keys
    k = np.zeros((1, 1, 2, D), np.float32)
    k[0, 0, 1, 0] = -0.875
    v = np.zeros((1, 1, 2, D), np.float32)
    v[0, 0, 0] = 1.0
    v[0, 0, 1] = -2.0
    mx = oracle.MxInputs.from_bf16(bf(q), bf(k), bf(v), 0, 2)
    out = oracle.attn_floor(mx, 2, False, 1.0, 2, [0])
    assert np.allclose(out[0], (1.0 - 0.75) / 1.375, atol=1e-12)


def test_emulate_with_exact_exp_equals_floor_on_one_tile():
    """On a single key tile the frozen maximum is the exact row maximum, so the
    emulation with the exact exp2 model (every mask bit set) takes the same codes as
    the exp-then-quantise floor and gives the same output; the cubic (no bit set)
    does not."""
    B, H, S, D = 1, 2, 128, 64
    rng = np.random.default_rng(5)
    q = bf(rng.standard_normal((B, H, S, D)) * 1.5)
    k, v = bf(rng.standard_normal((B, H, S, D))), bf(rng.standard_normal((B, H, S, D)))
    rows = allrows(B, H, S)
    for fq in (0, 1):
        mx = oracle.MxInputs.from_bf16(q, k, v, fq, fq)
        fl = oracle.attn_floor(mx, S, False, 0.125, fq, rows)
        hw = oracle.fsa_emulate(mx, S, False, 0.125, fq, rows, delta=8.0, mufu_mask=0xFFFFFFFF)["out"]
        po = oracle.fsa_emulate(mx, S, False, 0.125, fq, rows, delta=8.0, mufu_mask=0)["out"]
        assert np.array_equal(hw, fl), fq
        assert not np.array_equal(po, fl), fq


@pytest.mark.parametrize("a,b,phi,code_of_max", [(oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI, 7), (2.0, 2.0, 0.0, 6),
                                                 (2.0, 1.0, 0.0, 5), (1.5, 3.0, 0.75, 6)])
def test_emulate_efq_codes_span_the_e2m1_range(a, b, phi, code_of_max):
    """The EFQ rule maps onto the nonnegative E2M1 codes: over a few random rows every
    code from 0 up to the code of the row maximum occurs and none exceeds 7.  The
    score that sets the frozen maximum has t = 0 exactly, so its block exponent is
    E = floor(phi) - 2 = -2, its residual 2 and its code rne(2a + b) clamped to 7:
    rne(6.8125) = 7, rne(6) = 6, rne(5) = 5, rne(6) = 6 for the four rules."""
    B, H, S, D = 1, 1, 512, 64
    q, k, v = rnd((B, H, S, D), 1, 1.5), rnd((B, H, S, D), 2), rnd((B, H, S, D), 3)
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    rows = np.arange(0, S, 7, dtype=np.int64)
    res = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, delta=8.0, dump=True, efq_a=a, beta=b, phi=phi)
    pc = res["p_codes"]
    assert set(range(code_of_max + 1)) <= set(np.unique(pc)) <= set(range(8))
    for n in range(len(rows)):
        jmax = int(np.argmax(res["s"][n, :128]))     # the first tile's maximum sets M
        assert pc[n, jmax] == code_of_max


# --------------------------------------------------------------------------- exp2 approximation
def test_exp2_poly_exact_at_integers_and_error_bound():
    for n in range(-60, 10):
        assert oracle.exp2_poly(float(n)) == 2.0 ** n
    assert oracle.exp2_poly(-1000.0) == 2.0 ** -64           # clamp
    assert oracle.exp2_poly(float("-inf")) == 2.0 ** -64
    r = np.linspace(-20, 9.999, 20001, dtype=np.float32)
    p = np.array([oracle.exp2_poly(float(x)) for x in r])
    rel = np.abs(p / np.exp2(r.astype(np.float64)) - 1)
    assert rel.max() < 1.6e-4
    # interpolation nodes 1/3, 2/3 are met to fp32 rounding
    for f in (1 / 3, 2 / 3):
        assert abs(oracle.exp2_poly(float(np.float32(f))) / 2 ** float(np.float32(f)) - 1) < 1e-6


# --------------------------------------------------------------------------- emulation
FMTS = [(0, 0, 0), (1, 1, 1), (2, 2, 2), (2, 2, 3), (4, 4, 4)]      # (fmt_qk, fmt_v, fmt_p)


@pytest.mark.parametrize("fq,fv,fp", FMTS)
@pytest.mark.parametrize("mufu", [0, 0x55555555])
def test_emulate_zero_query_and_causal_row0(fq, fv, fp, mufu):
    B, H, S, D = 1, 1, 300, 128
    q0 = bf(np.zeros((B, H, S, D)))
    k, v = rnd((B, H, S, D), 2), rnd((B, H, S, D), 3)
    mx = oracle.MxInputs.from_bf16(q0, k, v, fq, fv)
    vh = oracle.decode_array(fv, mx.vc) * 2.0 ** (np.repeat(mx.vs.astype(np.int64), 32, -1) - 127)
    res = oracle.fsa_emulate(mx, S, True, 1 / math.sqrt(D), fp, allrows(B, H, S), mufu_mask=mufu)
    for i in (0, 1, 127, 128, 299):
        assert np.allclose(res["out"][i], vh[0, 0, :, :i + 1].mean(axis=1), atol=1e-12)
    assert not res["fallbacks"].any()
    assert np.array_equal(res["tiles"], np.arange(S) // 128 + 1)


@pytest.mark.parametrize("fq,fv,fp", FMTS)
def test_emulate_constant_v_is_one(fq, fv, fp):
    B, H, S, D = 1, 2, 257, 64
    q, k = rnd((B, H, S, D), 1), rnd((B, H, S, D), 2)
    ones = bf(np.ones((B, H, S, D)))
    mx = oracle.MxInputs.from_bf16(q, k, ones, fq, fv)
    res = oracle.fsa_emulate(mx, S, False, 0.125, fp, allrows(B, H, S))
    assert np.allclose(res["out"], 1.0, atol=1e-13)


def test_emulate_planted_score_fires_one_fallback():
    B, H, S, D = 1, 1, 384, 64
    rng = np.random.default_rng(0)
    q = rng.standard_normal((B, H, S, D)).astype(np.float32) * 0.1
    k = rng.standard_normal((B, H, S, D)).astype(np.float32) * 0.1
    k[0, 0, 7] = 2.0          # a key in the first tile that dominates every row's max
    q[0, 0, :, :] = np.abs(q[0, 0, :, :]) * np.sign(k[0, 0, 7])
    v = rnd((B, H, S, D), 3)
    rows = allrows(B, H, S)
    base = oracle.fsa_emulate(oracle.MxInputs.from_bf16(bf(q), bf(k), v, 0, 0), S, False, 0.125, 0, rows)
    assert not base["fallbacks"].any()
    k[0, 0, 300] = 8.0 * q[0, 0, 5] / np.abs(q[0, 0, 5]).max()   # large score for row 5, tile 2
    mx = oracle.MxInputs.from_bf16(bf(q), bf(k), v, 0, 0)
    res = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, dump=True)
    fired = np.nonzero(res["fallbacks"])[0]
    assert 5 in fired and res["fallbacks"][5] == 1
    mf = res["m_frozen"][5]
    assert mf[0] == mf[1] < mf[2]
    # a margin larger than the planted excess suppresses it; the output agrees to quantisation noise
    big = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, delta=40.0)
    assert not big["fallbacks"].any()
    ex = oracle.attn_floor(mx, S, False, 0.125, 0, rows, quantize_p=False)
    e_res = np.linalg.norm(res["out"] - ex) / np.linalg.norm(ex)
    e_big = np.linalg.norm(big["out"] - ex) / np.linalg.norm(ex)
    assert e_res < 0.1 and e_big < 0.1 and 0.5 < e_res / e_big < 2.0, (e_res, e_big)
    # a margin only moves the block exponents (the per-block scales absorb it): the
    # output stays within quantisation noise of the margin-free result
    d43 = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, delta=43.0)
    assert np.linalg.norm(d43["out"] - big["out"]) / np.linalg.norm(big["out"]) < 0.02


def test_emulate_pgen_block_structure():
    """Block max element gets the top codes; EFQ codes are a monotone function of
    the score within a block; integer residuals map to exact powers of two."""
    B, H, S, D = 1, 1, 256, 64
    q, k, v = rnd((B, H, S, D), 1, 1.5), rnd((B, H, S, D), 2), rnd((B, H, S, D), 3)
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    res = oracle.fsa_emulate(mx, S, False, 0.125, 3, allrows(B, H, S), dump=True)
    s, pc = res["s"], res["p_codes"]
    for row in range(0, S, 17):
        for b in range(S // 32):
            blk_s, blk_c = s[row, 32 * b:32 * b + 32], pc[row, 32 * b:32 * b + 32]
            assert blk_c[np.argmax(blk_s)] in (6, 7)
            order = np.argsort(blk_s, kind="stable")
            assert np.all(np.diff(blk_c[order].astype(int)) >= 0)
    mx8 = oracle.MxInputs.from_bf16(q, k, v, 0, 0)
    r8 = oracle.fsa_emulate(mx8, S, False, 0.125, 0, allrows(B, H, S), dump=True)
    top = {0x78, 0x7E}    # block max lands in [2^8, 448] (E4M3 256 .. 448)
    for row in range(0, S, 13):
        for b in range(S // 32):
            c = r8["p_codes"][row, 32 * b + np.argmax(r8["s"][row, 32 * b:32 * b + 32])]
            assert 0x78 <= c <= 0x7E


@pytest.mark.parametrize("fq,fp,bound", [(0, 0, 1.1), (1, 1, 1.1), (2, 2, 1.1), (2, 3, 1.17), (4, 4, 1.1),
                                           (5, 0, 1.1), (5, 3, 1.17)])
def test_emulate_error_close_to_floor_on_tiny(fq, fp, bound):
    """The pages' claim (Fused-Softmax brief, abstract): the approximation's extra
    error stays near the floor set by quantising the GEMM operands.  The exp paths
    meet 1.1x; the EFQ rule with the constants of oracle/efq_scan.py gives 1.114x on
    this case (the first reading a = b = 2, phi = 0 gave 1.51x), bounded at the EFQ
    tests' 1.17x."""
    from workloads import WORKLOADS, generate, sample_rows
    w = WORKLOADS["tiny"]
    q, k, v = generate(w)
    fv = 2 if fp == 3 else fp
    mx = oracle.MxInputs.from_bf16(q, k, v, fq, fv)
    rows = sample_rows(w)
    ex = oracle.attn_exact(q, k, v, w.causal, w.scale, rows)
    fl = oracle.attn_floor(mx, w.Sk, w.causal, w.scale, fv, rows)
    em = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows)["out"]
    e_fl = np.linalg.norm(fl - ex) / np.linalg.norm(ex)
    e_em = np.linalg.norm(em - ex) / np.linalg.norm(ex)
    assert e_em <= bound * e_fl, (e_em, e_fl)


# --------------------------------------------------------------------------- bf16 baseline emulation
def test_bf16_emulate_pins():
    B, H, S, D = 1, 2, 300, 64
    q, k, v = rnd((B, H, S, D), 1, 2.0), rnd((B, H, S, D), 2), rnd((B, H, S, D), 3)
    rows = allrows(B, H, S)
    z = oracle.bf16_emulate(bf(np.zeros((B, H, S, D))), k, v, True, 0.125, rows)["out"]
    vf = bf16_bits_to_f32(v).astype(np.float64)
    assert np.allclose(z[S + 200], vf[0, 1, :201].mean(axis=0), atol=1e-12)
    ones = oracle.bf16_emulate(q, k, bf(np.ones((B, H, S, D))), False, 0.125, rows)["out"]
    assert np.allclose(ones, 1.0, atol=1e-13)
    ex = oracle.attn_exact(q, k, v, True, 0.125, rows)
    em = oracle.bf16_emulate(q, k, v, True, 0.125, rows)["out"]
    assert np.abs(em - ex).max() / np.sqrt((ex ** 2).mean()) < 1e-2
    # growing scores across tiles trigger the lazy rescale only past tau
    kk = bf16_bits_to_f32(k).copy()
    kk[0, 0, 200] = 8.0 * bf16_bits_to_f32(q)[0, 0, 250]
    r = oracle.bf16_emulate(q, bf(kk), v, False, 0.125, rows)
    assert r["rescales"][250] == 1
    # the rescale keeps numerator and denominator consistent: still exact attention
    ex2 = oracle.attn_exact(q, bf(kk), v, False, 0.125, rows)
    assert np.abs(r["out"][250] - ex2[250]).max() / np.sqrt((ex2[250] ** 2).mean()) < 1e-2
    # without such a key, tile maxima move by far less than tau: no row rescales
    assert oracle.bf16_emulate(q, k, v, False, 0.125, rows)["rescales"].sum() == 0


def test_bf16_emulate_rounds_p_to_nearest_even():
    """p is rounded to bf16 with ties to even.  Scores 0 and s1 = -1.4140625 +
    0.0027770996 (exact in fp32) with c = fp32(scale log2 e) = 1: 2^s1 in fp32 is
    0.3759765625, exactly halfway between the bf16 neighbours 0.375 (even) and
    0.376953125, so p1 = 0.375 and, with v0 = 0 and v1 = 1, O = 0.375 / 1.375."""
    D = 64
    scale = float(np.float32(0.6931472))
    assert np.float32(np.float64(np.float32(scale)) * 1.4426950408889634) == 1.0
    a, b = np.float32(-1.4140625), np.float32(0.0027770996)
    s1 = np.float32(np.float64(a) + np.float64(b))
    assert np.float64(s1) == np.float64(a) + np.float64(b)
    assert np.float32(np.exp2(np.float64(s1))) == np.float32(0.3759765625)
    q = np.zeros((1, 1, 1, D), np.float32)
    q[..., :2] = 1.0
    k = np.zeros((1, 1, 2, D), np.float32)
    k[0, 0, 1, :2] = (a, b)
    v = np.zeros((1, 1, 2, D), np.float32)
    v[0, 0, 1] = 1.0
    assert np.array_equal(bf16_bits_to_f32(bf(k)), k)
    out = oracle.bf16_emulate(bf(q), bf(k), bf(v), False, scale, [0])["out"]
    assert np.allclose(out[0], 0.375 / 1.375, rtol=0, atol=1e-15)


def _one_query_case(kvals, D=64):
    """One query e_0 against keys k_j = kvals[j] e_0 (every value exact in bf16 and
    E4M3), scale fp32(ln 2) so that c = fp32(scale log2 e) = 1 and the log2-domain
    score of key j is kvals[j] exactly; V random integers."""
    S = len(kvals)
    q = np.zeros((1, 1, 1, D), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((1, 1, S, D), np.float32)
    k[0, 0, :, 0] = kvals
    v = np.random.default_rng(9).integers(-3, 4, (1, 1, S, D)).astype(np.float32)
    assert np.array_equal(bf16_bits_to_f32(bf(k)), k)
    scale = float(np.float32(0.6931472))
    assert np.float32(np.float64(np.float32(scale)) * 1.4426950408889634) == 1.0
    return oracle.MxInputs.from_bf16(bf(q), bf(k), bf(v), 0, 0), S, scale


def test_emulate_ambiguity_flags_boundary_cases():
    """The bound of undetermined decisions sees the two fp32 boundaries that a score
    perturbation of 2^-21 can cross.  Keys: tile 0 holds the maximum 0 (M = 0);
    (a) a block of tile 1 whose maximum is exactly -3, so its block exponent sits on
    floor's boundary: the bound is positive and covers the move when the scores
    grow by 2^-21 and the exponent drops by one; (b) a tile-1 key exactly at M +
    delta = 8: the fallback decision is undetermined, so the bound is infinite, and
    the perturbed run does fall back."""
    rng = np.random.default_rng(3)
    grid = np.array([-(1 + i / 8) * 2.0 ** e for i in range(8) for e in range(-1, 3)], np.float32)
    kv = rng.choice(grid[grid < -3.0], 256)
    kv[:128] = rng.choice(grid, 128)
    kv[0] = 0.0
    kv[128] = -3.0
    mx, S, scale = _one_query_case(kv)
    base = oracle.fsa_emulate(mx, S, False, scale, 0, [0], delta=8.0, mufu_mask=0xFFFFFFFF, ambiguity=True)
    pert = oracle.fsa_emulate(mx, S, False, scale, 0, [0], delta=8.0, mufu_mask=0xFFFFFFFF, s_perturb=2.0 ** -21)
    diff = np.abs(pert["out"] - base["out"])
    assert np.isfinite(base["amb"]).all() and base["amb"].max() > 0
    assert diff.max() > 0 and np.all(diff <= base["amb"] * (1 + 1e-9) + 1e-15)
    kv[130] = 8.0
    mx, S, scale = _one_query_case(kv)
    base = oracle.fsa_emulate(mx, S, False, scale, 0, [0], delta=8.0, mufu_mask=0xFFFFFFFF, ambiguity=True)
    pert = oracle.fsa_emulate(mx, S, False, scale, 0, [0], delta=8.0, mufu_mask=0xFFFFFFFF, s_perturb=2.0 ** -21)
    assert base["fallbacks"][0] == 0 and pert["fallbacks"][0] == 1
    assert np.isinf(base["amb"]).all()


@pytest.mark.parametrize("fq,fp,mufu", [(0, 0, 0xFFFFFFFF), (0, 0, 0), (2, 3, 0), (1, 2, 0x77777777)])
def test_emulate_ambiguity_bound_covers_score_perturbations(fq, fp, mufu):
    """amb bounds how far the output can move when the fp32 scores move within the
    modelled uncertainty: rerun the emulation with every score scaled by 1 +- 2^-21
    and 1 +- 2^-22 (coherently, inside the per-score interval) and check each change
    against the unperturbed bound.  The case is large enough that codes do flip."""
    w = small(WORKLOADS["prefill"], 1024, H=4, Hkv=2)
    w = Workload(w.name, w.B, w.H, w.Hkv, w.Sq, w.Sk, w.D, w.causal, ["E4M3", "E2M3", "E2M1"][fq],
                 ["E4M3", "E2M3", "E2M1", "E2M1_EFQ"][fp], w.seed, w.kind)
    q, k, v = generate(w)
    fv = 2 if fp == 3 else fp
    mx = oracle.MxInputs.from_bf16(q, k, v, fq, fv)
    rows = np.arange(w.B * w.H * w.Sq)
    base = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=8.0, mufu_mask=mufu, ambiguity=True)
    amb = base["amb"]
    assert np.all(amb >= 0.0)
    assert np.mean(np.isinf(amb).any(axis=1)) < 0.01
    moved = 0
    for eps in (2.0 ** -21, -2.0 ** -21, 2.0 ** -22, -2.0 ** -22):
        pert = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=8.0, mufu_mask=mufu, s_perturb=eps)
        diff = np.abs(pert["out"] - base["out"])
        moved += int(np.sum(diff.max(axis=1) > 1e-12))
        assert np.all(diff <= amb * (1 + 1e-9) + 1e-12), f"eps {eps}: {np.max(diff - amb):.3e}"
    assert moved > 0


# --------------------------------------------------------------------------- EFQ block scale and given scores
@pytest.mark.parametrize("a,b,phi", [(oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI), (1.5, 3.0, 0.75), (2.0, 2.0, 0.0)])
def test_emulate_efq_block_max_residual_window(a, b, phi):
    """E = floor(tmax + phi) - 2 puts every block's largest residual t - E in
    [2 - phi, 3 - phi), so the block maximum's code lies between the rule's codes at the
    two ends: rne(a (2 - phi) + b) .. rne(a (3 - phi) + b), clamped to 7; with phi > 0 the
    upper end is never reached by the OCP window [2, 3)."""
    B, H, S, D = 1, 1, 512, 64
    q, k, v = rnd((B, H, S, D), 11, 1.5), rnd((B, H, S, D), 12), rnd((B, H, S, D), 13)
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    rows = np.arange(0, S, 5, dtype=np.int64)
    res = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, delta=8.0, dump=True, efq_a=a, beta=b, phi=phi)
    lo = min(7, int(np.round(a * (2 - phi) + b)))
    hi = min(7, int(np.round(a * (3 - phi) + b)))
    seen = set()
    for n in range(len(rows)):
        for blk in range(S // 32):
            s = res["s"][n, 32 * blk:32 * blk + 32]
            c = int(res["p_codes"][n, 32 * blk + int(np.argmax(s))])
            assert lo <= c <= hi, (n, blk, c, lo, hi)
            seen.add(c)
    assert len(seen) >= 2


def test_emulate_phi_only_moves_efq_scales():
    """The reference point phi belongs to the EFQ rule: the exp-then-round paths keep
    the OCP block scale and give identical results for any phi; EFQ results change."""
    B, H, S, D = 1, 2, 300, 64
    q, k, v = rnd((B, H, S, D), 21), rnd((B, H, S, D), 22), rnd((B, H, S, D), 23)
    rows = allrows(B, H, S)
    for fq, fp in ((0, 0), (1, 1), (2, 2)):
        mx = oracle.MxInputs.from_bf16(q, k, v, fq, fp)
        r0 = oracle.fsa_emulate(mx, S, False, 0.125, fp, rows, phi=0.0, dump=True)
        r1 = oracle.fsa_emulate(mx, S, False, 0.125, fp, rows, phi=0.75, dump=True)
        assert np.array_equal(r0["p_codes"], r1["p_codes"]) and np.array_equal(r0["out"], r1["out"])
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    r0 = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, phi=0.0, dump=True)
    r1 = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, phi=0.75, dump=True)
    assert not np.array_equal(r0["p_scales"], r1["p_scales"])


def test_emulate_given_scores_drive_the_algorithm():
    """s_in replaces the emulation's own scores: given its own scores back, everything is
    unchanged (and no score uncertainty is left: for EFQ the ambiguity bound is zero on
    rows without a fallback, and the exp2 of a fallback's factor elsewhere);
    given a raised score in a late tile, that row falls back and its M follows it."""
    B, H, S, D = 1, 1, 384, 64
    q, k, v = rnd((B, H, S, D), 31), rnd((B, H, S, D), 32), rnd((B, H, S, D), 33)
    rows = allrows(B, H, S)
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    base = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, delta=0.0, dump=True)
    same = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, delta=0.0, dump=True, s_in=base["s"], ambiguity=True)
    for key in ("out", "p_codes", "p_scales", "fallbacks"):
        assert np.array_equal(base[key], same[key]), key
    # what is left is the hardware exp2 of a fallback's factor (2^-21 relative)
    nofb = same["fallbacks"] == 0
    assert nofb.any() and not same["amb"][nofb].any()
    assert np.all(same["amb"] <= 2.0 ** -20 * np.abs(same["out"]).max())
    s2 = base["s"].copy()
    row, key = 7, 300
    s2[row, key] = base["s"][row].max() + 40.0
    moved = oracle.fsa_emulate(mx, S, False, 0.125, 3, rows, delta=0.0, dump=True, s_in=s2)
    c = np.float32(np.float32(0.125) * np.float32(1.4426950408889634))
    assert moved["fallbacks"][row] == base["fallbacks"][row] + (0 if base["m_frozen"][row, 2] >= np.float32(s2[row, key] * c) else 1)
    assert moved["m_frozen"][row, 2] == np.float32(s2[row, key] * c)
    assert moved["p_codes"][row, key] == min(7, int(np.round(oracle.EFQ_A * 2 + oracle.EFQ_B)))


def test_emulate_given_codes_are_accumulated():
    """p_in replaces the P codes that are accumulated: the emulation's own codes back
    give the same output; zeroing the code of one key removes exactly that key's term,
    o' = (o l - p v) / (l - p), with p its decoded code times the block scale and l
    the row's sum of decoded P."""
    B, H, S, D = 1, 1, 128, 64
    q, k, v = rnd((B, H, S, D), 41), rnd((B, H, S, D), 42), rnd((B, H, S, D), 43)
    rows = allrows(B, H, S)
    mx = oracle.MxInputs.from_bf16(q, k, v, 0, 0)
    base = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, delta=8.0, dump=True)
    same = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, delta=8.0, dump=True, p_in=base["p_codes"])
    assert np.array_equal(base["out"], same["out"])
    row, key = 17, 40
    pc = base["p_codes"].copy()
    pc[row, key] = 0
    cut = oracle.fsa_emulate(mx, S, False, 0.125, 0, rows, delta=8.0, p_in=pc)
    sc = 2.0 ** (base["p_scales"][row].astype(np.int64) - 127)
    p = oracle.decode_array(0, base["p_codes"][row]) * np.repeat(sc, 32)
    l = p.sum()
    vh = oracle.decode_array(0, mx.vc[0, 0]) * 2.0 ** (np.repeat(mx.vs[0, 0].astype(np.int64), 32, -1) - 127)
    expect = (base["out"][row] * l - p[key] * vh[:, key]) / (l - p[key])
    assert np.allclose(cut["out"][row], expect, rtol=1e-12, atol=1e-15)
    others = np.arange(S) != row
    assert np.array_equal(cut["out"][others], base["out"][others])
