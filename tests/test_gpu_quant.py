"""Parity of the MX quantisation kernel (fsa_mx_quantize) with the oracle:
codes and scales bit-exact, on edge-case tensors and full workload shapes."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, generate, to_bf16_bits
from gpu_layout import unpack_rows, unpack_cols

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMTS = [0, 1, 2, 4]
ROW_FMTS = FMTS + [5]            # NVFP4 (fsa.h 5) is a rows (Q/K) format only


def _fsa():
    import softmax_mx_block_gb300 as fsa
    return fsa


def edge_tensor(shape, seed):
    """bf16 values mixing normals, exact rounding ties, zeros, signed zeros,
    subnormals, huge values and whole-zero / tiny blocks."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    flat = x.reshape(-1)
    pick = rng.random(flat.size)
    sel = pick < 0.1
    flat[sel] = rng.integers(-64, 64, sel.sum()) / 128.0       # ties of every format at block max 1.0
    flat[(pick >= 0.1) & (pick < 0.13)] = 0.0
    flat[(pick >= 0.13) & (pick < 0.15)] = -0.0
    sel = (pick >= 0.15) & (pick < 0.17)
    flat[sel] = rng.standard_normal(sel.sum()) * 1e-39           # bf16 subnormals
    sel = (pick >= 0.17) & (pick < 0.18)
    flat[sel] = rng.standard_normal(sel.sum()) * 1e30
    last = x.reshape(-1, shape[-1])
    for r in range(0, last.shape[0], 7):
        last[r, :32] = 0.0
    for r in range(3, last.shape[0], 11):
        last[r, :32] *= 1e-38
    if shape[-1] >= 64:
        for r in range(5, last.shape[0], 13):
            last[r, 32:64] = np.round(last[r, 32:64] * 4) / 4
            last[r, 32] = 2.0
    return to_bf16_bits(x)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _check_rows(x_bits, fmt):
    fsa = _fsa()
    B, H, S, D = x_bits.shape
    mt = fsa.fsa_mx_quantize(_dev(x_bits), fsa.FSA_MX_ROWS, fmt)
    torch.cuda.synchronize()
    c, s = unpack_rows(mt.codes.cpu().numpy(), mt.scales.cpu().numpy(), fmt, B, H, S, D)
    oc, os_ = oracle.mx_quantize_rows(x_bits, fmt)
    np.testing.assert_array_equal(s, os_)
    np.testing.assert_array_equal(c, oc)


def _check_cols(x_bits, fmt):
    fsa = _fsa()
    B, H, S, D = x_bits.shape
    mt = fsa.fsa_mx_quantize(_dev(x_bits), fsa.FSA_MX_COLS_T, fmt)
    torch.cuda.synchronize()
    c, s = unpack_cols(mt.codes.cpu().numpy(), mt.scales.cpu().numpy(), fmt, B, H, S, D)
    oc, os_ = oracle.mx_quantize_cols(x_bits, fmt)
    np.testing.assert_array_equal(s, os_)
    np.testing.assert_array_equal(c, oc)


@pytest.mark.parametrize("fmt", ROW_FMTS)
@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 77, 64), (1, 1, 1, 128), (1, 3, 129, 64)])
def test_quant_rows_edge(fmt, shape):
    _check_rows(edge_tensor(shape, 10 + fmt), fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 77, 64), (1, 1, 1, 128), (1, 2, 256, 64)])
def test_quant_cols_edge(fmt, shape):
    x = edge_tensor(shape, 20 + fmt)
    x[:, :, :32, ::5] = 0            # zero blocks along the sequence axis too
    _check_cols(x, fmt)


@pytest.mark.parametrize("fmt", ROW_FMTS)
def test_quant_nonfinite_block(fmt):
    x = np.random.default_rng(1).standard_normal((1, 1, 64, 128)).astype(np.float32)
    x[0, 0, 3, 40] = np.inf
    xb = to_bf16_bits(x)
    xb[0, 0, 9, 100] = 0x7FC0        # NaN
    _check_rows(xb, fmt)


@pytest.mark.parametrize("name", ["prefill", "long_efq_16k", "video_dit"])
def test_quant_full_workloads(name):
    w = WORKLOADS[name]
    q, k, v = generate(w)
    fq = {"E4M3": 0, "E2M3": 1, "E2M1": 2}[w.fmt_qk]
    fv = {"E4M3": 0, "E2M3": 1, "E2M1": 2, "E2M1_EFQ": 2}[w.fmt_pv]
    _check_rows(q, fq)
    _check_rows(k, fq)
    _check_cols(v, fv)


@pytest.mark.parametrize("fq,fv,B,H,Hkv,Sq,Sk,D", [
    (0, 0, 1, 4, 2, 300, 300, 128),      # GQA, ragged tail
    (1, 2, 1, 2, 2, 77, 200, 64),        # E2M3 / E2M1, rectangular, D 64
    (2, 2, 2, 3, 1, 129, 1, 128),        # one key
    (2, 0, 1, 1, 1, 512, 384, 64),
    (4, 4, 1, 2, 1, 300, 260, 128),      # E3M2 both
    (4, 2, 1, 2, 2, 100, 130, 64),
    (5, 2, 1, 4, 2, 300, 260, 128),      # NVFP4 Q/K, E2M1 V
    (5, 0, 2, 2, 1, 77, 129, 64),        # NVFP4 Q/K, E4M3 V, D 64
])
def test_quant_qkv_one_launch(fq, fv, B, H, Hkv, Sq, Sk, D):
    """The one-launch Q/K/V form writes the codes and scales of three separate
    calls, byte for byte (padding slots included), and those are the oracle's."""
    fsa = _fsa()
    q = edge_tensor((B, H, Sq, D), 30 + fq)
    k = edge_tensor((B, Hkv, Sk, D), 31 + fq)
    v = edge_tensor((B, Hkv, Sk, D), 32 + fv)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    mq, mk, mv = fsa.fsa_mx_quantize_qkv(qd, kd, vd, fq, fv)
    sq = fsa.fsa_mx_quantize(qd, fsa.FSA_MX_ROWS, fq)
    sk = fsa.fsa_mx_quantize(kd, fsa.FSA_MX_ROWS, fq)
    sv = fsa.fsa_mx_quantize(vd, fsa.FSA_MX_COLS_T, fv)
    torch.cuda.synchronize()
    for a, b in ((mq, sq), (mk, sk), (mv, sv)):
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    c, s_ = unpack_rows(mq.codes.cpu().numpy(), mq.scales.cpu().numpy(), fq, B, H, Sq, D)
    oc, os_ = oracle.mx_quantize_rows(q, fq)
    np.testing.assert_array_equal(s_, os_)
    np.testing.assert_array_equal(c, oc)
    c, s_ = unpack_cols(mv.codes.cpu().numpy(), mv.scales.cpu().numpy(), fv, B, Hkv, Sk, D)
    oc, os_ = oracle.mx_quantize_cols(v, fv)
    np.testing.assert_array_equal(s_, os_)
    np.testing.assert_array_equal(c, oc)


@pytest.mark.parametrize("layout", [0, 1])
def test_quant_padding_slots(layout):
    """Scale slots with no data hold 2^0 (0x7F): rows past S and blocks past D
    (rows layout), rows d >= D and key blocks past S (transposed layout)."""
    fsa = _fsa()
    B, H, S, D = 1, 2, 200, 64
    x = edge_tensor((B, H, S, D), 40)
    mt = fsa.fsa_mx_quantize(_dev(x), layout, 0)
    torch.cuda.synchronize()
    sc = mt.scales.cpu().numpy().reshape(B * H, -1, 512)
    r = np.arange(128)
    slot = lambda rr, b: (rr % 32) * 16 + (rr // 32) * 4 + b
    if layout == 0:
        for bh in range(B * H):
            assert (sc[bh, 0][slot(r, 2)] == 0x7F).all() and (sc[bh, 0][slot(r, 3)] == 0x7F).all()
            tail = r[r >= S - 128]
            for b in range(4):
                assert (sc[bh, 1][slot(tail, b)] == 0x7F).all()
    else:
        dd = r[r >= D]
        for bh in range(B * H):
            for t in range(2):
                for b in range(4):
                    assert (sc[bh, t][slot(dd, b)] == 0x7F).all()
            # block 3 of tile 1 (keys 224..255) lies wholly past S = 200
            for dv in range(D):
                assert sc[bh, 1][slot(dv, 3)] == 0x7F
