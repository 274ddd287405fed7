"""The C ABI library loads and exports every entry point include/fsa.h declares;
host-only calls (sizes, options, status strings, argument checks) work
without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = ""
    for name in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if name.endswith(".h"):
            src += open(os.path.join(ROOT, "include", name)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fsa_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import softmax_mx_block_gb300 as fsa
    return fsa.load()


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_sizes_and_status(lib):
    import softmax_mx_block_gb300 as fsa
    assert fsa.fsa_mx_sizes(1, 32, 4096, 128, fsa.FSA_MX_ROWS, "E4M3") == (32 * 4096 * 128, 32 * 32 * 512)
    assert fsa.fsa_mx_sizes(1, 32, 4096, 128, fsa.FSA_MX_ROWS, "E2M1") == (32 * 4096 * 64, 32 * 32 * 512)
    assert fsa.fsa_mx_sizes(1, 40, 75600, 128, fsa.FSA_MX_COLS_T, "E2M3") == (40 * 128 * 75648, 40 * 591 * 512)
    assert fsa.fsa_mx_sizes(1, 8, 300, 64, fsa.FSA_MX_COLS_T, "E2M1") == (8 * 64 * 384 // 2, 8 * 3 * 512)
    with pytest.raises(fsa.FsaError):
        fsa.fsa_mx_sizes(1, 1, 128, 96, 0, "E4M3")
    assert fsa.status_string(fsa.FSA_ERR_TIMEOUT) == "on-chip wait timed out"
    o = fsa.default_opts()
    assert (o.exp_mode, o.timeout_ms, o.delta, o.out_dtype) == (fsa.FSA_EXP_MUFU, 4000, 8.0, fsa.FSA_OUT_F32)
    assert not o.debug
    assert lib.fsa_version() == 200


def test_efq_defaults_match_the_oracle_reading(lib):
    """The EFQ rule's constants in the library's defaults are the ones the oracle
    uses (both follow the scan in oracle/efq_scan.py)."""
    import oracle
    import softmax_mx_block_gb300 as fsa
    o = fsa.default_opts()
    assert (o.efq_a, o.efq_b, o.efq_phi) == (oracle.EFQ_A, oracle.EFQ_B, oracle.EFQ_PHI)
    hdr = open(os.path.join(ROOT, "include", "fsa.h")).read()
    for name, val in (("A", oracle.EFQ_A), ("B", oracle.EFQ_B), ("PHI", oracle.EFQ_PHI)):
        m = re.search(rf"#define FSA_EFQ_{name}_DEFAULT\s+([0-9.]+)f", hdr)
        assert m and float(m.group(1)) == val


def test_argument_checks_reject_before_launch(lib):
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import fsa_mx_tensor
    t = fsa_mx_tensor(16, 16, 0, 0, 1, 1, 128, 128)
    v = fsa_mx_tensor(16, 16, 0, 1, 1, 1, 128, 128)
    vp = ctypes.c_void_p

    def args(q, k, vv, H, Hkv, D, fq, fp):
        return (ctypes.byref(q), ctypes.byref(k), ctypes.byref(vv), vp(16), 1, H, Hkv, 128, 128, D, 0,
                ctypes.c_float(0.125), fq, fp, vp(0))
    # H not a multiple of Hkv, D outside {64, 128}, EFQ as a QK format, null pointers
    assert lib.fsa_attention_fwd(*args(t, t, v, 3, 2, 128, 0, 0)) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_attention_fwd(*args(t, t, v, 1, 1, 96, 0, 0)) == fsa.FSA_ERR_INVALID_ARG
    # key length above 2^20 (the accuracy limit of fp32 accumulation in tensor memory)
    kl = fsa_mx_tensor(16, 16, 0, 0, 1, 1, (1 << 20) + 1, 128)
    vl = fsa_mx_tensor(16, 16, 0, 1, 1, 1, (1 << 20) + 1, 128)
    assert lib.fsa_attention_fwd(ctypes.byref(t), ctypes.byref(kl), ctypes.byref(vl), vp(16), 1, 1, 1, 128,
                                 (1 << 20) + 1, 128, 0, ctypes.c_float(0.125), 0, 0, vp(0)) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_attention_fwd(*args(t, t, v, 1, 1, 128, 3, 3)) == fsa.FSA_ERR_UNSUPPORTED_FMT
    assert lib.fsa_attention_fwd(None, None, None, vp(16), 1, 1, 1, 128, 128, 128, 0, ctypes.c_float(0.1), 0, 0,
                                 vp(0)) == fsa.FSA_ERR_INVALID_ARG
    # descriptor mismatch: V passed in the row layout
    assert lib.fsa_attention_fwd(*args(t, t, t, 1, 1, 128, 0, 0)) == fsa.FSA_ERR_INVALID_ARG
    # misaligned pointer
    bad = fsa_mx_tensor(17, 16, 0, 0, 1, 1, 128, 128)
    assert lib.fsa_attention_fwd(*args(bad, t, v, 1, 1, 128, 0, 0)) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_attention_fwd_bf16(vp(16), vp(16), vp(16), vp(16), 1, 2, 3, 128, 128, 128, 0,
                                      ctypes.c_float(0.1), vp(0), vp(0)) == fsa.FSA_ERR_INVALID_ARG
    x = fsa_mx_tensor(16, 16, 0, 0, 0, 0, 0, 0)
    assert lib.fsa_mx_quantize(vp(16), 1, 1, 128, 128, 0, 3, ctypes.byref(x), vp(0)) == fsa.FSA_ERR_UNSUPPORTED_FMT
    assert lib.fsa_mx_quantize(vp(0), 1, 1, 128, 128, 0, 0, ctypes.byref(x), vp(0)) == fsa.FSA_ERR_INVALID_ARG
    # the one-launch Q/K/V form: null or misaligned inputs, EFQ as a storage format, a bad head dimension
    ox, oy, oz = (fsa_mx_tensor(16, 16, 0, 0, 0, 0, 0, 0) for _ in range(3))

    def qkv(q, k, vv, D, fq, fv, o=ox):
        return lib.fsa_mx_quantize_qkv(q, k, vv, 1, 4, 2, 128, 256, D, fq, fv, ctypes.byref(o), ctypes.byref(oy),
                                       ctypes.byref(oz), vp(0))
    assert qkv(vp(16), vp(0), vp(16), 128, 0, 0) == fsa.FSA_ERR_INVALID_ARG
    assert qkv(vp(16), vp(24), vp(16), 128, 0, 0) == fsa.FSA_ERR_INVALID_ARG
    assert qkv(vp(16), vp(16), vp(16), 128, 0, 3) == fsa.FSA_ERR_UNSUPPORTED_FMT
    assert qkv(vp(16), vp(16), vp(16), 96, 0, 0) == fsa.FSA_ERR_INVALID_ARG
    assert qkv(vp(16), vp(16), vp(16), 128, 0, 0, o=fsa_mx_tensor(16, 0, 0, 0, 0, 0, 0, 0)) == fsa.FSA_ERR_INVALID_ARG


def test_kernel_poly_constants_match_oracle():
    """The exp2 cubic in the kernel source is the oracle's interpolant (same fp32 values)."""
    import oracle
    src = open(os.path.join(ROOT, "softmax_mx_block_gb300", "csrc", "fsa_attn.cu")).read()
    line = next(l for l in src.splitlines() if l.startswith("constexpr float kC3"))
    lits = [float.fromhex(x[:-1]) for x in re.findall(r"0x1\.[0-9a-f]+p-?\d+f", line)]
    c = oracle.exp2_poly_coeffs()
    assert sorted(lits) == sorted(float(x) for x in c[1:])


def test_binding_refuses_host_tensors(lib):
    """No CPU path: every compute entry of the binding rejects host tensors before
    any call into the library, instead of computing on the CPU."""
    import torch
    import softmax_mx_block_gb300 as fsa
    x = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16)
    with pytest.raises(fsa.FsaError, match="CUDA tensor"):
        fsa.fsa_mx_quantize(x, fsa.FSA_MX_ROWS, "E4M3")
    with pytest.raises(fsa.FsaError, match="CUDA tensor"):
        fsa.fsa_mx_quantize_qkv(x, x, x, "E4M3", "E4M3")
    with pytest.raises(fsa.FsaError, match="CUDA tensor"):
        fsa.fsa_attention_fwd_bf16(x, x, x)


def test_binding_checks_mx_buffers(lib):
    """The binding checks what the C ABI cannot see behind its bare pointers: MX
    buffers of the right dtype and at least fsa_mx_sizes bytes, on a CUDA device."""
    import torch
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import MxTensor, _check_mx_buffers, _need_mx
    B, H, S, D = 1, 2, 300, 64
    for layout, fmt in [(fsa.FSA_MX_ROWS, 0), (fsa.FSA_MX_ROWS, 2), (fsa.FSA_MX_COLS_T, 1), (fsa.FSA_MX_COLS_T, 2)]:
        cb, sb = fsa.fsa_mx_sizes(B, H, S, D, layout, fmt)
        ok = MxTensor(torch.empty(cb, dtype=torch.uint8), torch.empty(sb, dtype=torch.uint8), fmt, layout, B, H, S, D)
        _check_mx_buffers(ok, "t")
        for bad in (MxTensor(torch.empty(cb - 16, dtype=torch.uint8), ok.scales, fmt, layout, B, H, S, D),
                    MxTensor(ok.codes, torch.empty(sb - 1, dtype=torch.uint8), fmt, layout, B, H, S, D),
                    MxTensor(ok.codes.view(torch.int8), ok.scales, fmt, layout, B, H, S, D),
                    MxTensor(ok.codes, ok.scales, fmt, layout, B, H, S + 128, D)):
            with pytest.raises(fsa.FsaError):
                _check_mx_buffers(bad, "t")
        with pytest.raises(fsa.FsaError, match="CUDA tensor"):
            _need_mx(ok, "t", torch.device("cpu"))


def _attn_args(fsa, opts):
    from softmax_mx_block_gb300._binding import fsa_mx_tensor
    t = fsa_mx_tensor(16, 16, 0, 0, 1, 1, 128, 128)
    v = fsa_mx_tensor(16, 16, 0, 1, 1, 1, 128, 128)
    keep = (t, v, opts)
    return keep, (ctypes.byref(t), ctypes.byref(t), ctypes.byref(v), ctypes.c_void_p(16), 1, 1, 1, 128, 128, 128, 0,
                  ctypes.c_float(0.125), 0, 0, ctypes.byref(opts), ctypes.c_void_p(0), ctypes.c_void_p(0))


@pytest.mark.parametrize("field,value", [("delta", -1.0), ("delta", float("inf")), ("efq_a", 0.0), ("efq_a", 17.0),
                                         ("efq_b", 100.0), ("efq_phi", 1.0), ("efq_phi", -0.25), ("out_dtype", 2),
                                         ("exp_mode", 3), ("schedule", 5)])
def test_options_out_of_range_are_rejected(lib, field, value):
    """A negative margin (nearly every tile would fall back), EFQ constants outside
    their documented range, an unknown output dtype: INVALID_ARG before any launch."""
    import softmax_mx_block_gb300 as fsa
    o = fsa.default_opts()
    setattr(o, field, value)
    keep, a = _attn_args(fsa, o)
    assert lib.fsa_attention_fwd_ex(*a) == fsa.FSA_ERR_INVALID_ARG


def test_debug_dump_format_checks(lib):
    """The debug instance exists for the POLY / MUFU exp modes only; other requests,
    and dumps with a null buffer, are refused before any launch."""
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import fsa_debug_dump, fsa_mx_tensor
    d = fsa_debug_dump(16, 16, 16, 16)
    o = fsa.default_opts()
    o.debug = ctypes.pointer(d)
    t = fsa_mx_tensor(16, 16, 0, 0, 1, 1, 128, 128)
    v2 = fsa_mx_tensor(16, 16, 2, 1, 1, 1, 128, 128)
    args = (ctypes.byref(t), ctypes.byref(t), ctypes.byref(v2), ctypes.c_void_p(16), 1, 1, 1, 128, 128, 128, 0,
            ctypes.c_float(0.125), 0, 2, ctypes.byref(o), ctypes.c_void_p(0), ctypes.c_void_p(0))
    v0 = fsa_mx_tensor(16, 16, 0, 1, 1, 1, 128, 128)
    o.exp_mode = fsa.FSA_EXP_SPLIT
    args = (ctypes.byref(t), ctypes.byref(t), ctypes.byref(v0), ctypes.c_void_p(16), 1, 1, 1, 128, 128, 128, 0,
            ctypes.c_float(0.125), 0, 0, ctypes.byref(o), ctypes.c_void_p(0), ctypes.c_void_p(0))
    assert lib.fsa_attention_fwd_ex(*args) == fsa.FSA_ERR_UNSUPPORTED_FMT        # split exp mode
    d0 = fsa_debug_dump(16, 0, 16, 16)
    o.debug = ctypes.pointer(d0)
    o.exp_mode = fsa.FSA_EXP_MUFU
    assert lib.fsa_attention_fwd_ex(*args) == fsa.FSA_ERR_INVALID_ARG            # a null dump pointer


def test_layers_are_checked_before_any_launch(lib):
    """fsa_attention_fwd_layers checks every layer first: a bad later layer means no
    launch at all (the first layer's fake device pointers are never touched)."""
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import fsa_layer, fsa_mx_tensor
    t = fsa_mx_tensor(16, 16, 0, 0, 1, 1, 128, 128)
    v = fsa_mx_tensor(16, 16, 0, 1, 1, 1, 128, 128)
    arr = (fsa_layer * 2)()
    good = fsa_layer(ctypes.pointer(t), ctypes.pointer(t), ctypes.pointer(v), 16, 1, 1, 1, 128, 128, 128, 0, 0.125,
                     0, 0, 8.0, 0)
    arr[0] = good
    arr[1] = fsa_layer(ctypes.pointer(t), ctypes.pointer(t), ctypes.pointer(v), 16, 1, 1, 1, 128, 128, 128, 0, 0.125,
                       0, 0, -1.0, 0)                                          # negative margin
    assert lib.fsa_attention_fwd_layers(arr, 2, None, None) == fsa.FSA_ERR_INVALID_ARG
    arr[1] = fsa_layer(ctypes.pointer(t), ctypes.pointer(t), ctypes.pointer(v), 16, 1, 1, 1, 128, 128, 128, 0, 0.125,
                       0, 3, 8.0, 0)                                           # P format does not match V
    assert lib.fsa_attention_fwd_layers(arr, 2, None, None) == fsa.FSA_ERR_UNSUPPORTED_FMT
    assert lib.fsa_attention_fwd_layers(None, 1, None, None) == fsa.FSA_ERR_INVALID_ARG
    assert lib.fsa_attention_fwd_layers(None, 0, None, None) == fsa.FSA_OK


def test_tune_delta_host_logic(lib):
    """Layers whose fallback rate is above the target get a larger margin (capped);
    layers without evidence (timeout, no visited tiles) and quiet layers keep theirs."""
    import softmax_mx_block_gb300 as fsa
    st = [dict(fallback_events=50, row_tiles=1000, status=0),     # 5% > 1%: raise
          dict(fallback_events=5, row_tiles=1000, status=0),      # 0.5%: keep
          dict(fallback_events=900, row_tiles=1000, status=-4),   # timed out: no evidence
          dict(fallback_events=0, row_tiles=0, status=0),         # nothing visited
          dict(fallback_events=500, row_tiles=1000, status=0)]    # at the cap
    assert fsa.fsa_tune_delta(st, [8.0, 8.0, 8.0, 8.0, 62.0], 0.01, 4.0, 64.0) == [12.0, 8.0, 8.0, 8.0, 64.0]
    with pytest.raises(fsa.FsaError):
        fsa.fsa_tune_delta(st[:1], [70.0], 0.01, 4.0, 64.0)     # margin above the maximum
    with pytest.raises(fsa.FsaError):
        fsa.fsa_tune_delta(st[:1], [8.0], 0.01, 0.0, 64.0)      # no step


def test_mma_peak_argument_checks(lib):
    import softmax_mx_block_gb300 as fsa
    fl = ctypes.c_double()
    for kind, nn, n, it in ((4, 128, 1, 1), (-1, 128, 1, 1), (1, 64, 1, 1), (1, 128, 0, 1), (1, 256, 1, 0),
                            (1, 128, 70000, 1)):
        assert lib.fsa_mma_peak(kind, nn, n, it, None, ctypes.byref(fl), None) == fsa.FSA_ERR_INVALID_ARG


def test_nvfp4_is_a_rows_qk_format_with_two_scale_atoms(lib):
    """NVFP4 (fsa.h 5): Q/K rows only (D/64 scale atoms of 512 bytes per 128-row
    tile), never V or P; the attention call takes it as fmt_qk on one CTA per query
    tile with Q quantised beforehand, and refuses the persistent schedule and the
    prologue-quantised Q before any launch."""
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import fsa_mx_tensor
    assert fsa.fsa_mx_sizes(1, 32, 4096, 128, fsa.FSA_MX_ROWS, "NVFP4") == (32 * 4096 * 64, 32 * 32 * 1024)
    assert fsa.fsa_mx_sizes(1, 8, 300, 64, fsa.FSA_MX_ROWS, "NVFP4") == (8 * 300 * 32, 8 * 3 * 512)
    with pytest.raises(fsa.FsaError):
        fsa.fsa_mx_sizes(1, 8, 300, 128, fsa.FSA_MX_COLS_T, "NVFP4")
    vp = ctypes.c_void_p
    t = fsa_mx_tensor(16, 16, 5, 0, 1, 1, 128, 128)
    v = fsa_mx_tensor(16, 16, 5, 1, 1, 1, 128, 128)
    v2 = fsa_mx_tensor(16, 16, 2, 1, 1, 1, 128, 128)

    def args(q, vv, fq, fp, o):
        return (ctypes.byref(q), ctypes.byref(t), ctypes.byref(vv), vp(16), 1, 1, 1, 128, 128, 128, 0,
                ctypes.c_float(0.125), fq, fp, ctypes.byref(o), vp(0), vp(0))
    o = fsa.default_opts()
    assert lib.fsa_attention_fwd_ex(*args(t, v, 5, 5, o)) == fsa.FSA_ERR_UNSUPPORTED_FMT     # NVFP4 as PV
    o.schedule = 2                     # FSA_SCHED_PERSISTENT
    assert lib.fsa_attention_fwd_ex(*args(t, v2, 5, 2, o)) == fsa.FSA_ERR_UNSUPPORTED_FMT
    o = fsa.default_opts()
    assert lib.fsa_attention_fwd_qbf16(vp(16), ctypes.byref(t), ctypes.byref(v2), vp(16), 1, 1, 1, 128, 128, 128,
                                       0, ctypes.c_float(0.125), 5, 2, ctypes.byref(o), vp(0),
                                       vp(0)) == fsa.FSA_ERR_UNSUPPORTED_FMT
    x = fsa_mx_tensor(16, 16, 0, 0, 0, 0, 0, 0)
    assert lib.fsa_mx_quantize(vp(16), 1, 1, 128, 128, 1, 5, ctypes.byref(x), vp(0)) == fsa.FSA_ERR_INVALID_ARG


def test_host_entry_argument_checks(lib):
    """fsa_attention_fwd_host checks every argument before it creates a stream or
    enqueues a copy, so these calls need no GPU."""
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import fsa_device_io, fsa_host_io, fsa_mx_tensor
    vp = ctypes.c_void_p
    mq, mk, mv = (fsa_mx_tensor(16, 16, 0, 0, 0, 0, 0, 0) for _ in range(3))
    host = fsa_host_io(16, 16, 16, 16)

    def dev(q=16, out=16, m=mq):
        return fsa_device_io(q, 16, 16, ctypes.pointer(m), ctypes.pointer(mk), ctypes.pointer(mv), out)

    def call(h, d, H=4, Hkv=2, D=128, fq=0, fp=0, opts=None):
        return lib.fsa_attention_fwd_host(ctypes.byref(h) if h is not None else None,
                                          ctypes.byref(d) if d is not None else None, 1, H, Hkv, 256, 256, D, 1,
                                          ctypes.c_float(0.088), fq, fp,
                                          ctypes.byref(opts) if opts is not None else None, vp(0), 0, vp(0))
    assert call(None, dev()) == fsa.FSA_ERR_INVALID_ARG
    assert call(host, None) == fsa.FSA_ERR_INVALID_ARG
    assert call(fsa_host_io(16, 0, 16, 16), dev()) == fsa.FSA_ERR_INVALID_ARG          # null host k
    assert call(host, dev(q=24)) == fsa.FSA_ERR_INVALID_ARG                            # misaligned device q
    assert call(host, dev(m=fsa_mx_tensor(16, 0, 0, 0, 0, 0, 0, 0))) == fsa.FSA_ERR_INVALID_ARG
    assert call(host, dev(), H=3, Hkv=2) == fsa.FSA_ERR_INVALID_ARG                    # H not a multiple of Hkv
    assert call(host, dev(), D=96) == fsa.FSA_ERR_INVALID_ARG
    assert call(host, dev(), fq=3, fp=3) == fsa.FSA_ERR_UNSUPPORTED_FMT                 # EFQ as a QK^T format
    o = fsa.default_opts()
    o.delta = -1.0
    assert call(host, dev(), opts=o) == fsa.FSA_ERR_INVALID_ARG
    o = fsa.default_opts()
    dd = fsa._binding.fsa_debug_dump(16, 16, 16, 16, 0)
    o.debug = ctypes.pointer(dd)
    assert call(host, dev(), opts=o) == fsa.FSA_ERR_INVALID_ARG                        # no debug dumps here
