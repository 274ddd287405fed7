"""The host-memory entry point (fsa_attention_fwd_host): copies in, quantisation,
attention and copies back by groups of kv heads, the copies on streams of their own.
Every head runs the same kernels on the same data as in the device entry points, so
the output must equal theirs bit for bit for every chunking, and so must the
statistics and per-row fallback counts; one case is also checked against the oracle
the way the device path is."""
import numpy as np
import pytest

from workloads import WORKLOADS, generate, sample_rows, small

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from test_gpu_attention import FMT, check, oracle_mx, run_mx  # noqa: E402


def _host(bits, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t


def run_host(w, q, k, v, n_chunks, pinned=True, out_dtype=None, **kw):
    import softmax_mx_block_gb300 as fsa
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    stats = fsa.new_stats()
    rf = torch.zeros((w.B, w.H, w.Sq), dtype=torch.int32, device="cuda")
    out = fsa.fsa_attention_fwd_host(_host(q, pinned), _host(k, pinned), _host(v, pinned), fmt_qk=fq, fmt_pv=fp,
                                     causal=w.causal, scale=w.scale, n_chunks=n_chunks, stats=stats,
                                     row_fallbacks=rf, out_dtype=out_dtype, **kw)
    torch.cuda.current_stream().synchronize()
    return dict(out=out, stats=fsa.read_stats(stats), row_fallbacks=rf.cpu().numpy().reshape(-1))


# (workload, Sq, Sk, B, H, Hkv): four kv-head units over two batches, ragged lengths
CASES = [("long_fp8_16k", 700, 700, 2, 8, 2), ("long_efq_16k", 520, 1100, 2, 8, 2),
         ("video_dit", 400, 400, 1, 6, 6), ("long_nvfp4_16k", 300, 900, 2, 4, 2)]


@pytest.mark.parametrize("name,Sq,Sk,B,H,Hkv", CASES, ids=[c[0] for c in CASES])
def test_host_entry_matches_device_path(name, Sq, Sk, B, H, Hkv):
    w = small(WORKLOADS[name], Sq, Sk, H=H, Hkv=Hkv, B=B)
    q, k, v = generate(w)
    ref = run_mx(w, q, k, v, exp_mode=None, delta=None, row_fb=True)
    assert ref["stats"]["status"] == 0
    for n_chunks in (1, 3, 0, B * Hkv):
        got = run_host(w, q, k, v, n_chunks)
        assert got["stats"] == ref["stats"], n_chunks
        assert np.array_equal(got["row_fallbacks"], ref["row_fallbacks"]), n_chunks
        o = got["out"].numpy().reshape(-1, w.D)
        assert np.array_equal(o.view(np.uint32), ref["out"].view(np.uint32)), f"{name}: {n_chunks} chunks differ"


def test_host_entry_pageable_memory_and_bf16_output():
    import softmax_mx_block_gb300 as fsa
    w = small(WORKLOADS["long_efq_16k"], 384, 640, H=4, Hkv=2, B=1)
    q, k, v = generate(w)
    fq, fp = FMT[w.fmt_qk], FMT[w.fmt_pv]
    dq, dk, dv = (_host(a).cuda() for a in (q, k, v))
    mq, mk, mv = fsa.fsa_mx_quantize_qkv(dq, dk, dv, fq, 2 if fp == 3 else fp)
    ref = fsa.fsa_attention_fwd(mq, mk, mv, causal=w.causal, scale=w.scale, fmt_qk=fq, fmt_pv=fp, out_dtype="bf16")
    got = run_host(w, q, k, v, 2, pinned=False, out_dtype="bf16")
    assert got["out"].dtype == torch.bfloat16 and got["stats"]["status"] == 0
    assert torch.equal(got["out"].view(torch.int16), ref.view(torch.int16).cpu())


def test_host_entry_against_the_oracle():
    w = small(WORKLOADS["long_efq_16k"], 600, 600, H=4, Hkv=2, B=1)
    q, k, v = generate(w)
    got = run_host(w, q, k, v, 2)
    rows = sample_rows(w, per_head=48)
    orc = oracle_mx(w, q, k, v, rows, 0xFFFFFFFF, delta=8.0)
    check(w, dict(out=got["out"].numpy().reshape(-1, w.D), stats=got["stats"]), orc, rows, floor_ratio=1.18)
