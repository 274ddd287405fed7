"""P~ codes, block scales and the frozen maximum of the fused kernel against the
oracle's step-by-step P generation, bit for bit, given the kernel's own scores.

The EFQ-Softmax page (abstract) makes the nonnegative E2M1 codes under
exponent-only block scales the method's product; the Fused-Softmax digest ("Read
it as") freezes the row maximum with a fallback.  The tensor core's fp32 scores
are the one input the oracle cannot reproduce bit for bit (their accumulation
order is not specified), so the debug instance of the kernel dumps, for every
key tile, the raw scores it loaded, the frozen maximum M it used, and the P~ code
and scale words it wrote to tensor memory; the oracle replays the algorithm's
steps 2-4 on those scores (oracle.fsa_emulate(s_in=...)).  M, the scale bytes and
the codes must then agree exactly: EFQ and the cubic exp2 are bit-reproducible;
at hardware-exp2 positions the code may also be the one at the other end of the
exp2's documented uncertainty (p_alt), and nothing else.  The scores themselves
are checked against the oracle's exactly rounded ones within 2^-21 of the sum of
the absolute 32-element block products."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, Workload, generate, sample_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from test_gpu_attention import FMT, _dev  # noqa: E402

MASK = {0: 0x00000000, 1: 0xFFFFFFFF}          # exp mode -> hardware-exp2 positions


def _codes_from_words(words, fmt_pv):
    """[R, nkt, 32] uint32 words -> [R, nkt*128] codes in key order."""
    b = np.ascontiguousarray(words.astype(np.uint32)).view(np.uint8).reshape(words.shape[0], words.shape[1], 128)
    if fmt_pv in ("E4M3", "E2M3", "E3M2"):
        return b.reshape(words.shape[0], -1)
    nib = b[:, :, :64]
    return np.stack([nib & 0x0F, nib >> 4], axis=-1).reshape(words.shape[0], -1)


def run_debug(w: Workload, q, k, v, exp_mode, delta, rows=None, mx_dev=None):
    """The debug instance on the sampled rows (all rows when rows is None); returns the
    output (fp32 numpy [rows, D] of every row), the dump and the stats."""
    import softmax_mx_block_gb300 as fsa
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    fv = 2 if fp == 3 else fp
    if mx_dev is None:
        mx_dev = (fsa.fsa_mx_quantize(_dev(q), fsa.FSA_MX_ROWS, fq), fsa.fsa_mx_quantize(_dev(k), fsa.FSA_MX_ROWS, fq),
                  fsa.fsa_mx_quantize(_dev(v), fsa.FSA_MX_COLS_T, fv))
    mq, mk, mv = mx_dev
    dump = fsa.DebugDump(w.B, w.H, w.Sq, w.Sk, rows=rows)
    stats = fsa.new_stats()
    rf = torch.zeros((w.B, w.H, w.Sq), dtype=torch.int32, device="cuda")
    out = fsa.fsa_attention_fwd(mq, mk, mv, causal=w.causal, scale=w.scale, fmt_qk=fq, fmt_pv=fp,
                                exp_mode=exp_mode, delta=delta, stats=stats, debug=dump, row_fallbacks=rf)
    torch.cuda.synchronize()
    st = fsa.read_stats(stats)
    assert st["status"] == 0
    return out, dump, st, rf


def compare_pgen(w: Workload, q, k, v, exp_mode, delta, rows, dump, mx=None, score_rows=None, outputs=False):
    """Checks the dumped M, scale bytes and codes of the sampled rows against the
    oracle's replay on the dumped scores (after checking those scores against the
    oracle's exactly rounded ones, on the first `score_rows` rows, all by default).
    With outputs=True also replays the accumulation on the kernel's own codes (once
    they are checked) and returns that output with its ambiguity bound (left: the
    hardware exp2 of a fallback's factor)."""
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    if mx is None:
        mx = oracle.MxInputs.from_bf16(q, k, v, fq, 2 if fp == 3 else fp)
    skp = (w.Sk + 31) // 32 * 32
    nkt = (w.Sk + 127) // 128
    s_gpu = dump.s.cpu().numpy()[:, :skp]
    m_gpu = dump.m.cpu().numpy()
    p_gpu = _codes_from_words(dump.p.cpu().numpy(), w.fmt_pv)
    sf_gpu = dump.p_scales.cpu().numpy().astype(np.uint32).view(np.uint8).reshape(len(rows), -1)
    mask = MASK[exp_mode] if fp != 3 else 0
    # the kernel's scores against the oracle's exactly rounded ones (a valid result of
    # the unspecified fp32 accumulation order: within 2^-21 of the block partial sums)
    ns = len(rows) if score_rows is None else min(score_rows, len(rows))
    own = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows[:ns], delta=delta, mufu_mask=mask, dump=True)
    vis = np.isfinite(own["s"])
    assert np.array_equal(vis, np.isfinite(s_gpu[:ns])), "masked keys differ"
    ds = np.abs(s_gpu[:ns][vis] - own["s"][vis])
    assert ds.max() <= 1e-5 * np.abs(own["s"][vis]).max() + 1e-6
    del own
    given = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=delta, mufu_mask=mask, dump=True,
                               s_in=s_gpu)
    # frozen maximum of every visited tile, bit for bit
    seen = ~np.isnan(given["m_frozen"])
    assert np.array_equal(m_gpu[:, :nkt][seen].view(np.uint32), given["m_frozen"][seen].view(np.uint32))
    # scale bytes of every 32-key block
    assert np.array_equal(sf_gpu[:, :skp // 32], given["p_scales"])
    # codes: exact, or the other end of the hardware exp2's uncertainty
    pg = p_gpu[:, :skp]
    exact = pg == given["p_codes"]
    alt_ok = pg == given["p_alt"]
    assert np.all(exact | alt_ok), f"{int(np.sum(~(exact | alt_ok)))} codes outside the allowed set"
    if exp_mode == 0 or fp == 3:
        assert np.all(exact)
    res = dict(n_alt=int(np.sum(~exact)), n=int(exact.size), given=given)
    if outputs:
        res["replay"] = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=delta, mufu_mask=mask,
                                           s_in=s_gpu, p_in=pg, ambiguity=True)
    return res


def check_pgen(w: Workload, q, k, v, exp_mode, delta, rows):
    out, dump, st, rf = run_debug(w, q, k, v, exp_mode, delta, rows=rows)
    res = compare_pgen(w, q, k, v, exp_mode, delta, rows, dump)
    # per-row fallback counts, given the same scores, exactly
    assert np.array_equal(rf.cpu().numpy().reshape(-1)[rows], res["given"]["fallbacks"])
    return res


SMALL = [
    (Workload("pg_e4m3", 1, 2, 1, 256, 300, 64, False, "E4M3", "E4M3", 31), 1, 0.0),
    (Workload("pg_e4m3_poly_causal", 1, 2, 2, 384, 384, 128, True, "E4M3", "E4M3", 32, "k_outliers"), 0, 8.0),
    (Workload("pg_e2m3", 1, 2, 1, 256, 520, 128, False, "E2M3", "E2M3", 33, "planted"), 0, 0.0),
    (Workload("pg_e2m3_mufu", 1, 2, 1, 256, 520, 128, False, "E2M3", "E2M3", 33, "planted"), 1, 8.0),
    (Workload("pg_e2m1", 1, 2, 2, 300, 300, 128, True, "E2M1", "E2M1", 34), 0, 0.0),
    (Workload("pg_e2m1_mufu", 1, 2, 2, 300, 300, 64, True, "E2M1", "E2M1", 34), 1, 8.0),
    (Workload("pg_efq", 1, 4, 2, 512, 1024, 128, True, "E2M1", "E2M1_EFQ", 35, "planted"), 1, 0.0),
    (Workload("pg_efq_d64", 1, 2, 1, 200, 700, 64, False, "E2M1", "E2M1_EFQ", 36), 1, 8.0),
    (Workload("pg_e3m2", 1, 2, 1, 256, 520, 128, True, "E3M2", "E3M2", 38, "planted"), 0, 0.0),
    (Workload("pg_e3m2_mufu", 1, 2, 1, 300, 300, 64, False, "E3M2", "E3M2", 39), 1, 8.0),
    (Workload("pg_nvfp4_efq", 1, 4, 2, 384, 700, 128, True, "NVFP4", "E2M1_EFQ", 40, "planted"), 1, 0.0),
    (Workload("pg_nvfp4_e4m3_d64", 1, 2, 1, 256, 300, 64, False, "NVFP4", "E4M3", 41), 0, 8.0),
]


@pytest.mark.parametrize("w,exp_mode,delta", SMALL, ids=[c[0].name for c in SMALL])
def test_pgen_bit_exact_given_kernel_scores(w, exp_mode, delta):
    q, k, v = generate(w)
    rows = np.arange(w.B * w.H * w.Sq, dtype=np.int64)
    res = check_pgen(w, q, k, v, exp_mode, delta, rows)
    # the debug instance dumps all rows the same way when no row selection is given
    import softmax_mx_block_gb300 as fsa  # noqa: F401
    out_all, dump_all, _, _ = run_debug(w, q, k, v, exp_mode, delta)
    assert torch.equal(dump_all.s.cpu(), run_debug(w, q, k, v, exp_mode, delta, rows=rows)[1].s.cpu())
    if exp_mode == 1 and w.fmt_pv != "E2M1_EFQ":
        assert res["n_alt"] <= 1e-3 * res["n"]          # the exp2 uncertainty touches few codes


def test_pgen_planted_fallbacks_fire():
    """With delta = 0 on planted keys the dumped M rises across tiles (fallbacks) and
    still matches the oracle's replay bit for bit."""
    w = Workload("pg_planted", 1, 2, 2, 256, 1024, 128, False, "E2M1", "E2M1_EFQ", 37, "planted")
    q, k, v = generate(w)
    res = check_pgen(w, q, k, v, 1, 0.0, np.arange(w.B * w.H * w.Sq, dtype=np.int64))
    assert res["given"]["fallbacks"].sum() > 0


@pytest.mark.parametrize("name,exp_mode", [("tiny", 0), ("tiny", 1), ("prefill", 1), ("long_efq_16k", 1)])
def test_pgen_full_length_tiles(name, exp_mode):
    """The workloads' own sizes: every tile of the sampled rows (64 per head)."""
    w = WORKLOADS[name]
    q, k, v = generate(w)
    check_pgen(w, q, k, v, exp_mode, 8.0, sample_rows(w, per_head=64))
