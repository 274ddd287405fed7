"""The library's further entry points on the GPU, through the C ABI: bf16 output,
the per-layer (hybrid-format) schedule call, margin tuning from device stats, and
the tensor-core peak probe."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, Workload, generate, sample_rows, small

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from test_gpu_attention import FMT, TOL_EMU, _dev, oracle_mx  # noqa: E402


def _fsa():
    import softmax_mx_block_gb300 as fsa
    return fsa


def _mx(w, q, k, v):
    fsa = _fsa()
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    fv = 2 if fp == 3 else fp
    return (fsa.fsa_mx_quantize(_dev(q), fsa.FSA_MX_ROWS, fq), fsa.fsa_mx_quantize(_dev(k), fsa.FSA_MX_ROWS, fq),
            fsa.fsa_mx_quantize(_dev(v), fsa.FSA_MX_COLS_T, fv))


def _bf16_rne_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> 16) & 1)) >> 16).astype(np.uint16)


BF16_CASES = [
    (Workload("bf16out_e4m3", 1, 4, 2, 300, 300, 128, True, "E4M3", "E4M3", 41), 1),
    (Workload("bf16out_e4m3_pers", 1, 4, 2, 300, 300, 128, True, "E4M3", "E4M3", 41), 2),
    (Workload("bf16out_efq_d64", 1, 2, 1, 256, 700, 64, False, "E2M1", "E2M1_EFQ", 42), 1),
    (Workload("bf16out_efq_d64_pers", 1, 2, 1, 256, 700, 64, False, "E2M1", "E2M1_EFQ", 42), 2),
    (Workload("bf16out_e2m3_nokeys", 1, 3, 3, 700, 300, 128, True, "E2M3", "E2M1", 43), 2),
]


@pytest.mark.parametrize("w,schedule", BF16_CASES, ids=[c[0].name for c in BF16_CASES])
def test_bf16_output_is_the_rounded_fp32_output(w, schedule):
    """out_dtype bf16 writes the same fp32 quotients rounded to nearest even: bit for bit
    the RNE of the fp32 output, under both schedules; against the oracle's emulation the
    tolerance grows by the bf16 rounding, |O - O_emu| <= (2e-3 rms + amb)(1 + 2^-8) +
    2^-8 |O_emu| (bf16 keeps 8 significant bits, so rounding moves a value by at most
    2^-8 of it; amb is the oracle's bound of what fp32 scores leave undetermined)."""
    fsa = _fsa()
    q, k, v = generate(w)
    mq, mk, mv = _mx(w, q, k, v)
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    kw = dict(causal=w.causal, scale=w.scale, fmt_qk=fq, fmt_pv=fp, schedule=schedule)
    o32 = fsa.fsa_attention_fwd(mq, mk, mv, **kw)
    o16 = fsa.fsa_attention_fwd(mq, mk, mv, out_dtype="bf16", **kw)
    torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    b16 = o16.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, w.D)
    f32 = o32.cpu().numpy().reshape(-1, w.D)
    assert np.array_equal(b16, _bf16_rne_bits(f32))
    rows = sample_rows(w)
    mx = oracle.MxInputs.from_bf16(q, k, v, fq, 2 if fp == 3 else fp)
    orc = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, fp, rows, delta=8.0, mufu_mask=0xFFFFFFFF, ambiguity=True)
    emu, amb = orc["out"], orc["amb"]
    det = ~np.isinf(amb).any(axis=1)
    o = (b16.astype(np.uint32) << 16).view(np.float32)[rows]
    # the fp32 output's bound (2e-3 rms plus what fp32 leaves undetermined), then the rounding
    tol = (TOL_EMU * np.sqrt(np.mean(emu ** 2)) + amb) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(emu)
    assert np.all((np.abs(o - emu) <= tol)[det])
    assert det.mean() > 0.99


def test_layer_schedule_matches_single_calls():
    """fsa_attention_fwd_layers runs each layer with its own formats and margin: outputs
    and per-layer stats equal those of one fsa_attention_fwd call per layer."""
    fsa = _fsa()
    base = small(WORKLOADS["adversarial"], 512, H=2, B=1)
    layers, singles = [], []
    deltas = [0.0, 8.0, 4.0, 16.0]
    for l in range(4):
        wl = base.layer(l)
        q, k, v = generate(wl)
        mq, mk, mv = _mx(wl, q, k, v)
        st = fsa.new_stats()
        layers.append(dict(q=mq, k=mk, v=mv, causal=wl.causal, scale=wl.scale, fmt_qk=wl.fmt_qk,
                           fmt_pv=wl.fmt_pv, delta=deltas[l], stats=st))
        st1 = fsa.new_stats()
        singles.append((fsa.fsa_attention_fwd(mq, mk, mv, causal=wl.causal, scale=wl.scale, fmt_qk=FMT[wl.fmt_qk],
                                              fmt_pv=FMT[wl.fmt_pv], delta=deltas[l], stats=st1), st1))
    outs = fsa.fsa_attention_fwd_layers(layers)
    torch.cuda.synchronize()
    for l, (o, (o1, st1)) in enumerate(zip(outs, singles)):
        assert torch.equal(o.view(torch.int32), o1.view(torch.int32)), l
        assert fsa.read_stats(layers[l]["stats"]) == fsa.read_stats(st1)
    # margin tuning from the layers' device stats: layers above the target rate get more
    rates = [fsa.read_stats(L["stats"]) for L in layers]
    new = fsa.fsa_tune_delta(rates, deltas, target_rate=1e-3, step=4.0, max_delta=64.0)
    for r, d0, d1 in zip(rates, deltas, new):
        above = r["row_tiles"] and r["fallback_events"] / r["row_tiles"] > 1e-3
        assert d1 == (min(64.0, d0 + 4.0) if above else d0)
    assert rates[0]["fallback_events"] > 0                  # delta 0 on planted keys falls back


@pytest.mark.parametrize("n", [128, 256])
@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_mma_peak_probe_runs(kind, n):
    """The throughput probe completes without a timeout on every SM and reports a
    plausible rate (a few hundred TFLOP/s at least for a short launch)."""
    fsa = _fsa()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fsa.fsa_mma_peak(kind, n_sm, 200, status, n=n)            # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flops = fsa.fsa_mma_peak(kind, n_sm, 20000, status, n=n)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert 200.0 < tflops < 30000.0, tflops


FUSED_Q_CASES = [
    Workload("fq_e4m3_causal", 1, 4, 2, 300, 300, 128, True, "E4M3", "E4M3", 51, "k_outliers"),
    Workload("fq_e2m3_d64", 1, 2, 1, 256, 700, 64, False, "E2M3", "E2M1", 52),
    Workload("fq_efq", 1, 4, 2, 520, 1100, 128, True, "E2M1", "E2M1_EFQ", 53),
    Workload("fq_efq_d64_rect", 1, 3, 3, 700, 300, 64, True, "E2M1", "E2M1_EFQ", 54),
    Workload("fq_e2m1_e4m3", 2, 2, 2, 200, 200, 128, False, "E2M1", "E4M3", 55),
    Workload("fq_e3m2", 1, 2, 2, 300, 400, 128, True, "E3M2", "E3M2", 56),
]


@pytest.mark.parametrize("w", FUSED_Q_CASES, ids=lambda w: w.name)
def test_fused_q_quantisation_is_bit_identical(w):
    """fsa_attention_fwd_qbf16 quantises bf16 Q in the attention kernel's prologue: the
    output, per-row fallback counts and stats equal those of quantising Q with
    fsa_mx_quantize first, bit for bit (ragged tails, rows without keys, both head
    dimensions, every QK^T format)."""
    fsa = _fsa()
    q, k, v = generate(w)
    mq, mk, mv = _mx(w, q, k, v)
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    kw = dict(causal=w.causal, scale=w.scale, fmt_qk=fq, fmt_pv=fp, schedule=1)
    res = []
    for qq in (mq, _dev(q)):
        st = fsa.new_stats()
        rf = torch.zeros((w.B, w.H, w.Sq), dtype=torch.int32, device="cuda")
        o = fsa.fsa_attention_fwd(qq, mk, mv, stats=st, row_fallbacks=rf, **kw)
        torch.cuda.synchronize()
        res.append((o, fsa.read_stats(st), rf))
    assert torch.equal(res[0][0].view(torch.int32), res[1][0].view(torch.int32))
    assert res[0][1] == res[1][1] and torch.equal(res[0][2], res[1][2])
    assert res[1][1]["status"] == 0


def test_fused_q_refuses_unsupported_options():
    fsa = _fsa()
    w = FUSED_Q_CASES[0]
    q, k, v = generate(w)
    _, mk, mv = _mx(w, q, k, v)
    for kw in (dict(schedule=2), dict(exp_mode=0)):
        with pytest.raises(fsa.FsaError, match="unsupported"):
            fsa.fsa_attention_fwd(_dev(q), mk, mv, causal=True, fmt_qk=0, fmt_pv=0, **kw)
