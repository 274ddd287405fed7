"""Parity of the MX quantisation kernel (fsa_mx_quantize) with the oracle:
codes and scales bit-exact, on edge-case tensors and full workload shapes."""
import numpy as np
import pytest

import oracle
from workloads import WORKLOADS, generate, to_bf16_bits
from gpu_layout import unpack_rows, unpack_cols

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FMTS = [0, 1, 2]


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


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 77, 64), (1, 1, 1, 128), (1, 3, 129, 64)])
def test_quant_rows_edge(fmt, shape):
    _check_rows(edge_tensor(shape, 10 + fmt), fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 1, 77, 64), (1, 1, 1, 128), (1, 2, 256, 64)])
def test_quant_cols_edge(fmt, shape):
    x = edge_tensor(shape, 20 + fmt)
    x[:, :, :32, ::5] = 0            # zero blocks along the sequence axis too
    _check_cols(x, fmt)


@pytest.mark.parametrize("fmt", FMTS)
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
