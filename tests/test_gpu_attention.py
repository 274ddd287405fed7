"""Parity of the fused MX attention kernel (fsa_attention_fwd_ex) and the BF16
kernel (fsa_attention_fwd_bf16) with the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, Workload, generate, sample_rows, small, to_bf16_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMT = {"E4M3": 0, "E2M3": 1, "E2M1": 2, "E2M1_EFQ": 3, "E3M2": 4, "NVFP4": 5}
SPLIT_MASK = 0x77777777          # key positions 4k+3 use the cubic, the rest the hardware exp2
TOL_EMU = 2e-3                   # max |O - O_emu| / rms(O_emu)
# error vs fp64 exact over the error of exact softmax with the same MX operands (the
# floor): 1.1 for the exp-then-round paths; for the EFQ direct codes the largest ratio
# the chosen rule reaches on the parity cases plus 5%, by QK^T format: E2M1 1.121
# (300 keys, non-causal, margin 8), E3M2 1.159 (300 keys, margin 0)
FLOOR_EXP = 1.1
FLOOR_EFQ = {"E2M1": 1.18, "E3M2": 1.22, "NVFP4": 1.18}


def _fsa():
    import softmax_mx_block_gb300 as fsa
    return fsa


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run_mx(w: Workload, q, k, v, exp_mode=2, delta=0.0, row_fb=False, **kw):
    fsa = _fsa()
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    fv = 2 if fp == 3 else fp
    mq = fsa.fsa_mx_quantize(_dev(q), fsa.FSA_MX_ROWS, fq)
    mk = fsa.fsa_mx_quantize(_dev(k), fsa.FSA_MX_ROWS, fq)
    mv = fsa.fsa_mx_quantize(_dev(v), fsa.FSA_MX_COLS_T, fv)
    stats = fsa.new_stats()
    rf = torch.zeros((w.B, w.H, w.Sq), dtype=torch.int32, device="cuda") if row_fb else None
    out = fsa.fsa_attention_fwd(mq, mk, mv, causal=w.causal, scale=w.scale, fmt_qk=fq, fmt_pv=fp,
                                exp_mode=exp_mode, delta=delta, row_fallbacks=rf, stats=stats, **kw)
    torch.cuda.synchronize()
    res = dict(out=out.cpu().numpy().reshape(-1, w.D), stats=fsa.read_stats(stats))
    if row_fb:
        res["row_fallbacks"] = rf.cpu().numpy().reshape(-1)
    return res


def oracle_mx(w, q, k, v, rows, mask, delta=0.0, with_floor=True):
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    fv = 2 if fp == 3 else fp
    mx = oracle.MxInputs.from_bf16(q, k, v, fq, fv)
    emu = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=delta, mufu_mask=mask, ambiguity=True)
    res = dict(emu=emu["out"], fallbacks=emu["fallbacks"], tiles=emu["tiles"], amb=emu["amb"])
    if with_floor:
        res["floor"] = oracle.attn_floor(mx, w.Sk, w.causal, w.scale, fv, rows)
        res["exact"] = oracle.attn_exact(q, k, v, w.causal, w.scale, rows)
    return res


def rel_err(a, ref):
    return np.linalg.norm(a - ref) / np.linalg.norm(ref)


def check(w, gpu, orc, rows, floor_ratio=FLOOR_EXP):
    """|O - O_emu| <= 2e-3 rms, plus, where the hardware exp2 (whose result the oracle
    brackets, not reproduces) may land a code on the other side of a rounding boundary,
    the oracle's bound of what that can change (amb).  At most 1% of the elements may
    need that slack.  Rows whose fallback decision fp32 leaves undetermined (amb
    infinite) get no slack."""
    o = gpu["out"][rows]
    emu = orc["emu"]
    rms = np.sqrt(np.mean(emu ** 2))
    d = np.abs(o - emu)
    amb = orc.get("amb", np.zeros_like(emu))
    slack = np.where(np.isfinite(amb), amb, 0.0)
    assert np.all(d <= TOL_EMU * rms + slack), f"{w.name}: max|O-O_emu|/rms = {d.max() / rms:.3e}"
    beyond = d > TOL_EMU * rms
    assert beyond.mean() <= 0.01, f"{w.name}: {int(beyond.sum())} elements beyond 2e-3 rms"
    if "exact" in orc and floor_ratio is not None:
        e_gpu, e_floor = rel_err(o, orc["exact"]), rel_err(orc["floor"], orc["exact"])
        assert e_gpu <= floor_ratio * e_floor, f"{w.name}: error {e_gpu:.4f} vs floor {e_floor:.4f}"
    assert gpu["stats"]["status"] == 0


def test_tiny_config_all_rows():
    w = WORKLOADS["tiny"]
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v)
    orc = oracle_mx(w, q, k, v, rows, SPLIT_MASK)
    check(w, gpu, orc, rows)
    assert gpu["stats"]["fallback_events"] == int(orc["fallbacks"].sum())
    assert gpu["stats"]["row_tiles"] == int(orc["tiles"].sum())


PAIRS = [("E4M3", "E4M3"), ("E2M3", "E2M1"), ("E2M1", "E2M1_EFQ"), ("E2M3", "E2M3"), ("E2M1", "E2M1"),
         ("E4M3", "E2M1"), ("E2M1", "E4M3"), ("E3M2", "E3M2"), ("E3M2", "E2M1_EFQ"), ("E2M3", "E3M2"),
         ("NVFP4", "E2M1_EFQ"), ("NVFP4", "E4M3"), ("NVFP4", "E2M1")]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("fq,fp", PAIRS)
def test_small_formats(fq, fp, D, causal):
    w = Workload(f"small_{fq}_{fp}_{D}_{int(causal)}", 1, 4, 2, 300, 300, D, causal, fq, fp, 5)
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v, row_fb=True)
    orc = oracle_mx(w, q, k, v, rows, SPLIT_MASK)
    ratio = FLOOR_EFQ[fq] if fp == "E2M1_EFQ" else FLOOR_EXP
    check(w, gpu, orc, rows, ratio)
    assert np.array_equal(gpu["row_fallbacks"][rows], orc["fallbacks"])


@pytest.mark.parametrize("fq,fp", [("E4M3", "E4M3"), ("E2M1", "E2M1_EFQ")])
def test_batched_causal_gqa(fq, fp):
    """Several batches and kv heads under the causal block order (one kv head per slow
    grid index, query tiles heaviest first with the query heads of a tile together):
    every (batch, head, query tile) is computed once and lands in its own rows."""
    w = Workload(f"batched_{fq}_{fp}", 3, 6, 2, 520, 520, 128, True, fq, fp, 31)
    q, k, v = generate(w)
    rows = sample_rows(w, per_head=64)
    gpu = run_mx(w, q, k, v, row_fb=True)
    orc = oracle_mx(w, q, k, v, rows, SPLIT_MASK)
    check(w, gpu, orc, rows, FLOOR_EFQ[fq] if fp == "E2M1_EFQ" else FLOOR_EXP)
    assert np.array_equal(gpu["row_fallbacks"][rows], orc["fallbacks"])


@pytest.mark.parametrize("exp_mode,mask", [(0, 0), (1, 0xFFFFFFFF), (2, SPLIT_MASK)])
def test_exp_modes(exp_mode, mask):
    w = small(WORKLOADS["prefill"], 384, H=4, Hkv=2)
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v, exp_mode=exp_mode)
    check(w, gpu, oracle_mx(w, q, k, v, rows, mask), rows)


@pytest.mark.parametrize("fq,fp,exp_mode,mask", [("E4M3", "E4M3", 2, SPLIT_MASK), ("E2M3", "E2M1", 1, 0xFFFFFFFF),
                                                 ("E3M2", "E3M2", 1, 0xFFFFFFFF), ("E2M1", "E2M1", 0, 0),
                                                 ("E2M1", "E2M1_EFQ", 1, 0)])
def test_rectangular_causal_and_empty_rows(fq, fp, exp_mode, mask):
    """Sq > Sk with causal bottom-right alignment: the first Sq - Sk queries see no key
    and get zero rows, also when they share a query tile with rows that have keys (a
    row whose frozen maximum is still -inf must produce zero codes in every format)."""
    w = Workload("rect", 1, 2, 1, 300, 200, 128, True, fq, fp, 9)
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v, exp_mode=exp_mode)
    orc = oracle_mx(w, q, k, v, rows, mask, with_floor=False)
    empty = [r for r in rows if (r % w.Sq) < w.Sq - w.Sk]
    assert np.all(gpu["out"][empty] == 0.0)
    check(w, gpu, orc, rows)


def test_fallback_counts_adversarial_small():
    w = small(WORKLOADS["adversarial"], 1024, H=3, B=1)
    for layer in (0, 1):
        wl = w.layer(layer)
        q, k, v = generate(wl)
        rows = sample_rows(wl)
        gpu = run_mx(wl, q, k, v, row_fb=True)
        orc = oracle_mx(wl, q, k, v, rows, SPLIT_MASK, with_floor=False)
        check(wl, gpu, orc, rows)
        fb_gpu = gpu["row_fallbacks"][rows]
        assert orc["fallbacks"].sum() > 0
        # the decision compares fp32 scores; allow rare one-ulp ties to differ
        assert np.mean(fb_gpu != orc["fallbacks"]) < 0.01
        assert gpu["stats"]["fallback_events"] == int(gpu["row_fallbacks"].sum())


def test_margin_delta():
    w = small(WORKLOADS["adversarial"], 512, H=2, B=1).layer(0)
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v, delta=6.0, row_fb=True)
    orc = oracle_mx(w, q, k, v, rows, SPLIT_MASK, delta=6.0, with_floor=False)
    check(w, gpu, orc, rows)


@pytest.mark.parametrize("name", ["tiny", "prefill", "adversarial"])
def test_default_margin(name):
    """The library default (frozen-max margin 8 log2 units) against the oracle at the same margin."""
    w = WORKLOADS[name]
    w = w if name == "tiny" else small(w, 640, H=4, Hkv=2 if name == "prefill" else None, B=1)
    w = w.layer(1) if w.layers > 1 else w
    q, k, v = generate(w)
    rows = sample_rows(w)
    gpu = run_mx(w, q, k, v, delta=None, row_fb=True)
    orc = oracle_mx(w, q, k, v, rows, SPLIT_MASK, delta=8.0)
    check(w, gpu, orc, rows)
    assert np.mean(gpu["row_fallbacks"][rows] != orc["fallbacks"]) < 0.01


@pytest.mark.parametrize("schedule", [1, 2])
def test_inject_stall_times_out_and_context_survives(schedule):
    fsa = _fsa()
    w = WORKLOADS["tiny"]
    q, k, v = generate(w)
    gpu = run_mx(w, q, k, v, inject_stall=True, timeout_ms=50, schedule=schedule)
    assert gpu["stats"]["status"] == fsa.FSA_ERR_TIMEOUT
    again = run_mx(w, q, k, v, schedule=schedule)
    assert again["stats"]["status"] == 0 and np.isfinite(again["out"]).all()


# ----------------------------------------------------------------------------- BF16 kernel
def run_bf16(w, q, k, v):
    fsa = _fsa()
    vt = fsa.fsa_bf16_transpose_v(_dev(v))
    stats = fsa.new_stats()
    out = fsa.fsa_attention_fwd_bf16(_dev(q), _dev(k), vt, causal=w.causal, scale=w.scale, stats=stats)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(-1, w.D), fsa.read_stats(stats)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_kernel(D, causal):
    w = Workload("bf16", 1, 4, 2, 300, 300, D, causal, "E4M3", "E4M3", 7)
    q, k, v = generate(w)
    rows = sample_rows(w)
    out, st = run_bf16(w, q, k, v)
    emu = oracle.bf16_emulate(q, k, v, causal, w.scale, rows)["out"]
    ex = oracle.attn_exact(q, k, v, causal, w.scale, rows)
    o = out[rows]
    assert np.abs(o - emu).max() / np.sqrt(np.mean(emu ** 2)) < 5e-3
    assert rel_err(o, ex) < 1e-2
    assert st["status"] == 0


def test_bf16_transpose_v():
    fsa = _fsa()
    v = to_bf16_bits(np.random.default_rng(2).standard_normal((2, 3, 200, 64)).astype(np.float32))
    vt = fsa.fsa_bf16_transpose_v(_dev(v))
    torch.cuda.synchronize()
    got = vt.cpu().view(torch.int16).numpy().view(np.uint16)
    assert got.shape == (2, 3, 64, 256)
    np.testing.assert_array_equal(got[..., :200], np.swapaxes(v, 2, 3))
    assert not got[..., 200:].any()


# the library's constants (codes never above 7: the kernel skips the fix of code 8)
# at margins 8 and 0, and with a margin above 120 (the fix path); other rules on both
# sides of a (3 - phi) + b < 7.49
EFQ_RULES = [(oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI, 8.0), (oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI, 0.0),
             (oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI, 200.0), (1.6875, 3.5, 0.5625, 8.0),
             (2.0, 2.0, 0.0, 8.0), (2.0, -3.0, 0.0, 8.0), (1.5, 3.0, 0.75, 120.0), (3.0, 5.5, 0.25, 50.0),
             (2.0, 2.0, 0.0, 200.0)]


@pytest.mark.parametrize("a,b,phi,delta", EFQ_RULES)
def test_efq_rule_constants_and_margin(a, b, phi, delta):
    """EFQ codes clamp(rne(a r + b), 0, 7) under E = floor(tmax + phi) - 2, for the
    library's constants and others (codes clamped at either end, large fallback
    margins that leave the block exponent far above the frozen maximum), on inputs with
    planted keys that lift late tiles far above it."""
    w = Workload("efq_rule", 1, 4, 2, 512, 1024, 128, False, "E2M1", "E2M1_EFQ", 11, "planted")
    q, k, v = generate(w)
    rows = sample_rows(w, per_head=128)
    gpu = run_mx(w, q, k, v, exp_mode=None, delta=delta, efq_a=a, efq_b=b, efq_phi=phi)
    assert gpu["stats"]["status"] == 0
    mx = oracle.MxInputs.from_bf16(q, k, v, FMT[w.fmt_qk], 2)
    orc = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, 3, rows, delta=delta, beta=b, efq_a=a, phi=phi,
                             ambiguity=True)
    emu, amb = orc["out"], orc["amb"]
    undetermined = np.isinf(amb).any(axis=1)
    assert np.mean(undetermined) < 0.01
    tol = TOL_EMU * np.sqrt(np.mean(emu ** 2))
    excess = (np.abs(gpu["out"][rows] - emu) - amb - tol)[~undetermined]
    assert np.all(excess <= 0.0), f"rule {(a, b, phi)} delta {delta}: exceeds by {excess.max():.3e}"


SCHED_CASES = [
    Workload("sched_ragged", 1, 4, 2, 300, 700, 128, False, "E4M3", "E4M3", 21),
    Workload("sched_causal_d64", 2, 4, 1, 640, 640, 64, True, "E2M3", "E2M1", 22),
    Workload("sched_no_keys", 1, 3, 3, 700, 300, 128, True, "E2M1", "E2M1_EFQ", 23),   # query tiles without key tiles
    Workload("sched_planted", 1, 2, 2, 1024, 1024, 128, True, "E4M3", "E4M3", 24, "planted"),
]


@pytest.mark.parametrize("w", SCHED_CASES, ids=lambda w: w.name)
def test_schedules_bit_identical(w):
    """One CTA per query tile and the persistent schedule run the same arithmetic per
    key tile: outputs, per-row fallback counts and statistics agree bit for bit."""
    q, k, v = generate(w)
    res = [run_mx(w, q, k, v, exp_mode=None, delta=None, row_fb=True, schedule=s) for s in (1, 2)]
    for r in res:
        assert r["stats"]["status"] == 0
    assert np.array_equal(res[0]["out"].view(np.uint32), res[1]["out"].view(np.uint32))
    assert np.array_equal(res[0]["row_fallbacks"], res[1]["row_fallbacks"])
    assert res[0]["stats"] == res[1]["stats"]


def test_persistent_more_query_tiles_than_one_wave():
    """More than 256 query tiles per SM: the persistent launch takes enough CTAs that
    none walks more than 256, and still matches one CTA per query tile bit for bit."""
    fsa = _fsa()
    g = torch.Generator(device="cuda").manual_seed(5)
    B, H, Hkv, S, Sk, D = 4, 80, 1, 16384, 256, 64          # 40960 query tiles
    x = lambda *shape: torch.randn(*shape, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = x(B, H, S, D), x(B, Hkv, Sk, D), x(B, Hkv, Sk, D)
    mq = fsa.fsa_mx_quantize(q, fsa.FSA_MX_ROWS, 0)
    mk = fsa.fsa_mx_quantize(k, fsa.FSA_MX_ROWS, 0)
    mv = fsa.fsa_mx_quantize(v, fsa.FSA_MX_COLS_T, 0)
    outs = []
    for s in (1, 2):
        st = fsa.new_stats()
        outs.append(fsa.fsa_attention_fwd(mq, mk, mv, fmt_qk=0, fmt_pv=0, stats=st, schedule=s))
        torch.cuda.synchronize()
        assert fsa.read_stats(st)["status"] == 0
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))


@pytest.mark.parametrize("causal", [False, True])
def test_head_count_at_the_grid_limit(causal):
    """B*H = 65535, the most the attention calls accept (one grid axis carries the
    heads, or the kv heads when causal): every head lands in its own rows.  Six heads
    spread over the range, the first and the last included, are checked against the
    oracle on all their rows (the heads are independent, so they form a small call of
    their own for the oracle)."""
    fsa = _fsa()
    B, H, S, D = 1, 65535, 130, 64
    g = torch.Generator(device="cuda").manual_seed(11)
    x = lambda: torch.randn(B, H, S, D, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = x(), x(), x()
    mq, mk, mv = fsa.fsa_mx_quantize_qkv(q, k, v, "E4M3", "E4M3")
    st = fsa.new_stats()
    out = fsa.fsa_attention_fwd(mq, mk, mv, causal=causal, scale=D ** -0.5, fmt_qk=0, fmt_pv=0, exp_mode=1,
                                delta=8.0, stats=st)
    torch.cuda.synchronize()
    assert fsa.read_stats(st)["status"] == 0
    heads = [0, 1, 4097, 32768, 65533, 65534]
    bits = lambda t: t[0, heads].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)[None]
    w = Workload("grid_limit", 1, len(heads), len(heads), S, S, D, causal, "E4M3", "E4M3", 11)
    rows = np.arange(len(heads) * S, dtype=np.int64)
    orc = oracle_mx(w, bits(q), bits(k), bits(v), rows, 0xFFFFFFFF, delta=8.0, with_floor=False)
    gpu = dict(out=out[0, heads].cpu().numpy().reshape(-1, D), stats=fsa.read_stats(st))
    check(w, gpu, orc, rows, None)
    del q, k, v, mq, mk, mv, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fq,fp", [("E2M1", "E2M1_EFQ"), ("E4M3", "E4M3")])
@pytest.mark.parametrize("causal", [False, True])
def test_longest_key_length(causal, fq, fp):
    """Sk = 2^20, the longest key length the attention calls accept: 8192 key tiles per
    query tile, every key and byte offset at its largest.  The first and last rows of
    both query tiles of two query heads sharing one kv head are checked against the
    oracle.  (The limit is set by accuracy: the fp32 accumulator in tensor memory
    drifts by a per-row factor that grows with the key tiles added into it; at 2^20
    keys it stays within the parity bound, at 2^22 it does not for 8-bit P~.)"""
    fsa = _fsa()
    B, H, Hkv, Sq, Sk, D = 1, 2, 1, 130, 1 << 20, 64
    g = torch.Generator(device="cuda").manual_seed(12)
    x = lambda h, s: torch.randn(B, h, s, D, generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = x(H, Sq), x(Hkv, Sk), x(Hkv, Sk)
    fv = "E2M1" if fp == "E2M1_EFQ" else fp
    mq, mk, mv = fsa.fsa_mx_quantize_qkv(q, k, v, fq, fv)
    st = fsa.new_stats()
    out = fsa.fsa_attention_fwd(mq, mk, mv, causal=causal, scale=D ** -0.5, fmt_qk=fq, fmt_pv=fp, exp_mode=1,
                                delta=8.0, stats=st)
    torch.cuda.synchronize()
    assert fsa.read_stats(st)["status"] == 0
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    w = Workload(f"longest_keys_{fq}_{fp}", B, H, Hkv, Sq, Sk, D, causal, fq, fp, 12)
    rows = np.array([0, 127, 128, 129, Sq, Sq + 127, Sq + 128, Sq + 129], dtype=np.int64)
    orc = oracle_mx(w, bits(q), bits(k), bits(v), rows, 0xFFFFFFFF, delta=8.0, with_floor=False)
    gpu = dict(out=out.cpu().numpy().reshape(-1, D), stats=fsa.read_stats(st))
    check(w, gpu, orc, rows, None)
    del q, k, v, mq, mk, mv, out
    torch.cuda.empty_cache()
