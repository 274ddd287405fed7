"""CPU oracle for MX block-scaled attention with a reformulated softmax.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``softmax_mx_block_gb300``) never imports, links or
runs anything here, and this package shares no code with it.

The arithmetic lives in ``fsa_oracle.c`` (plain C, fp64, OpenMP over query
rows); this module only builds it with gcc and marshals numpy arrays.

Parity pins live in ``tests/test_oracle_*.py``.  Parity unpinned (the pages fix
neither): the exact form of the fast exp2 of the Fused-Softmax digest ("Read it
as") and the constants of the EFQ-Softmax affine rule (abstract); the readings
used here are documented in ``fsa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT = {"E4M3": 0, "E2M3": 1, "E2M1": 2, "E8M0": 3, "E2M1_EFQ": 3, "E3M2": 4, "NVFP4": 5}
EMAX = {0: 8, 1: 2, 2: 2, 4: 4}


def build(force: bool = False) -> str:
    """Compile fsa_oracle.c into oracle/_build/liboracle.so (gcc, no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        # -ffp-contract=off: the fp32 steps of the emulation are part of its
        # definition; a fused a*b+c where the source writes two operations
        # would change the rounding.
        cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("Hkv", ctypes.c_int), ("Sq", ctypes.c_int),
                ("Sk", ctypes.c_int), ("D", ctypes.c_int), ("causal", ctypes.c_int)]


class MxOperands(ctypes.Structure):
    _fields_ = [("qc", ctypes.c_void_p), ("qs", ctypes.c_void_p), ("kc", ctypes.c_void_p),
                ("ks", ctypes.c_void_p), ("vc", ctypes.c_void_p), ("vs", ctypes.c_void_p),
                ("fmt_qk", ctypes.c_int), ("fmt_v", ctypes.c_int)]


class FsaOpts(ctypes.Structure):
    _fields_ = [("delta", ctypes.c_float), ("mufu_mask", ctypes.c_uint32), ("beta", ctypes.c_float),
                ("efq_a", ctypes.c_float), ("phi", ctypes.c_float), ("s_perturb", ctypes.c_double)]


class FsaDump(ctypes.Structure):
    _fields_ = [("s", ctypes.c_void_p), ("p_codes", ctypes.c_void_p), ("p_scales", ctypes.c_void_p),
                ("m_frozen", ctypes.c_void_p), ("amb", ctypes.c_void_p), ("s_in", ctypes.c_void_p),
                ("p_alt", ctypes.c_void_p), ("p_in", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            L = _lib
            L.orc_decode.restype = ctypes.c_double
            L.orc_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
            L.orc_encode.restype = ctypes.c_uint32
            L.orc_encode.argtypes = [ctypes.c_int, ctypes.c_double]
            L.orc_exp2_poly.restype = ctypes.c_float
            L.orc_exp2_poly.argtypes = [ctypes.c_float]
            L.orc_max_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def nthreads_default() -> int:
    return int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1))


# --------------------------------------------------------------------------- codecs
def decode(fmt: int, code: int) -> float:
    return lib().orc_decode(int(fmt), int(code))


def encode(fmt: int, x: float) -> int:
    return int(lib().orc_encode(int(fmt), float(x)))


def decode_array(fmt: int, codes) -> np.ndarray:
    """Vector decode through a 256-entry table built from orc_decode."""
    table = np.array([decode(fmt, c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def exp2_poly(r: float) -> float:
    return float(lib().orc_exp2_poly(float(r)))


def exp2_poly_coeffs() -> np.ndarray:
    c = np.zeros(4, np.float32)
    lib().orc_exp2_poly_coeffs(_p(c))
    return c


# --------------------------------------------------------------------------- MX quantise
def mx_quantize_rows(x_bf16: np.ndarray, fmt: int, nthreads: int | None = None):
    """Blocks of 32 along the last axis.  x_bf16: uint16 [..., L].

    Returns (codes uint8 [..., Lp], scales uint8 [..., Lp/32]) with Lp = L rounded
    up to a multiple of 32 (padding codes 0).  fmt 5 (NVFP4): blocks of 16 with
    E4M3 scales, see nvfp4_quantize_rows."""
    if fmt == 5:
        return nvfp4_quantize_rows(x_bf16, nthreads)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    L = x.shape[-1]
    Lp = (L + 31) // 32 * 32
    nrows = int(np.prod(x.shape[:-1]))
    codes = np.zeros(x.shape[:-1] + (Lp,), np.uint8)
    scales = np.zeros(x.shape[:-1] + (Lp // 32,), np.uint8)
    lib().orc_mx_quantize(_p(x), ctypes.c_int64(nrows), ctypes.c_int64(L), ctypes.c_int64(L), ctypes.c_int64(1),
                          ctypes.c_int(fmt), _p(codes), ctypes.c_int64(Lp), _p(scales), ctypes.c_int64(Lp // 32),
                          ctypes.c_int(nthreads or nthreads_default()))
    return codes, scales


def nvfp4_quantize_rows(x_bf16: np.ndarray, nthreads: int | None = None):
    """NVFP4 (orc_nvfp4_quantize): blocks of 16 along the last axis, E2M1 codes and
    one E4M3 scale byte per block.  Returns (codes uint8 [..., Lp], scales uint8
    [..., Lp/16]), Lp = L rounded up to a multiple of 16."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    L = x.shape[-1]
    Lp = (L + 15) // 16 * 16
    nrows = int(np.prod(x.shape[:-1]))
    codes = np.zeros(x.shape[:-1] + (Lp,), np.uint8)
    scales = np.zeros(x.shape[:-1] + (Lp // 16,), np.uint8)
    lib().orc_nvfp4_quantize(_p(x), ctypes.c_int64(nrows), ctypes.c_int64(L), ctypes.c_int64(L), ctypes.c_int64(1),
                             _p(codes), ctypes.c_int64(Lp), _p(scales), ctypes.c_int64(Lp // 16),
                             ctypes.c_int(nthreads or nthreads_default()))
    return codes, scales


def mx_quantize_cols(x_bf16: np.ndarray, fmt: int, nthreads: int | None = None):
    """Blocks of 32 along axis -2 (the sequence axis of [B,H,S,D]).

    Returns the transposed logical layout: codes uint8 [B,H,D,Sp], scales
    uint8 [B,H,D,Sp/32], Sp = S rounded up to a multiple of 32."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    B, H, S, D = x.shape
    Sp = (S + 31) // 32 * 32
    codes = np.zeros((B, H, D, Sp), np.uint8)
    scales = np.zeros((B, H, D, Sp // 32), np.uint8)
    L = lib()
    for b in range(B):
        for h in range(H):
            xs = x[b, h]
            cs = codes[b, h]
            ss = scales[b, h]
            L.orc_mx_quantize(_p(xs), ctypes.c_int64(D), ctypes.c_int64(S), ctypes.c_int64(1), ctypes.c_int64(D),
                              ctypes.c_int(fmt), _p(cs), ctypes.c_int64(Sp), _p(ss), ctypes.c_int64(Sp // 32),
                              ctypes.c_int(nthreads or nthreads_default()))
    return codes, scales


# --------------------------------------------------------------------------- attention
def _geom(B, H, Hkv, Sq, Sk, D, causal):
    return Geom(int(B), int(H), int(Hkv), int(Sq), int(Sk), int(D), int(bool(causal)))


def _rows(rows):
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def attn_exact(q, k, v, causal, scale, rows, nthreads=None):
    """fp64 softmax(scale q k^T) v from raw bf16 (uint16) q [B,H,Sq,D], k/v [B,Hkv,Sk,D]."""
    q = np.ascontiguousarray(q, np.uint16); k = np.ascontiguousarray(k, np.uint16)
    v = np.ascontiguousarray(v, np.uint16)
    B, H, Sq, D = q.shape; Hkv, Sk = k.shape[1], k.shape[2]
    rows = _rows(rows)
    out = np.zeros((len(rows), D), np.float64)
    g = _geom(B, H, Hkv, Sq, Sk, D, causal)
    lib().orc_attn_exact(_p(q), _p(k), _p(v), ctypes.byref(g), ctypes.c_double(scale), _p(rows),
                         ctypes.c_int64(len(rows)), _p(out), ctypes.c_int(nthreads or nthreads_default()))
    return out


class MxInputs:
    """Logical MX operands: q/k codes+scales blocked along D, v transposed and blocked along keys."""

    def __init__(self, qc, qs, kc, ks, vc, vs, fmt_qk, fmt_v):
        self.qc, self.qs, self.kc, self.ks, self.vc, self.vs = [np.ascontiguousarray(a, np.uint8)
                                                                for a in (qc, qs, kc, ks, vc, vs)]
        self.fmt_qk, self.fmt_v = int(fmt_qk), int(fmt_v)

    def struct(self):
        return MxOperands(self.qc.ctypes.data, self.qs.ctypes.data, self.kc.ctypes.data, self.ks.ctypes.data,
                          self.vc.ctypes.data, self.vs.ctypes.data, self.fmt_qk, self.fmt_v)

    @staticmethod
    def from_bf16(q, k, v, fmt_qk, fmt_v, nthreads=None):
        qc, qs = mx_quantize_rows(q, fmt_qk, nthreads)
        kc, ks = mx_quantize_rows(k, fmt_qk, nthreads)
        vc, vs = mx_quantize_cols(v, fmt_v, nthreads)
        return MxInputs(qc, qs, kc, ks, vc, vs, fmt_qk, fmt_v)


def _shape(mx: MxInputs, Sk):
    B, H, Sq, D = mx.qc.shape
    Hkv = mx.kc.shape[1]
    return B, H, Hkv, Sq, Sk, D


def attn_floor(mx: MxInputs, Sk, causal, scale, fmt_p, rows, quantize_p=True, nthreads=None):
    """Exact softmax over dequantised MX operands, P optionally MX-quantised (exp-then-quantize)."""
    B, H, Hkv, Sq, _, D = _shape(mx, Sk)
    rows = _rows(rows)
    out = np.zeros((len(rows), D), np.float64)
    g = _geom(B, H, Hkv, Sq, Sk, D, causal)
    ops = mx.struct()
    lib().orc_attn_floor(ctypes.byref(ops), ctypes.byref(g), ctypes.c_double(scale), ctypes.c_int(fmt_p),
                         ctypes.c_int(int(quantize_p)), _p(rows), ctypes.c_int64(len(rows)), _p(out),
                         ctypes.c_int(nthreads or nthreads_default()))
    return out


EFQ_A, EFQ_B, EFQ_PHI = 1.6875, 3.4375, 0.625      # the EFQ rule's constants (see efq_scan.py)


def fsa_emulate(mx: MxInputs, Sk, causal, scale, fmt_p, rows, delta=0.0, mufu_mask=0, beta=EFQ_B,
                efq_a=EFQ_A, phi=EFQ_PHI, dump=False, ambiguity=False, s_perturb=0.0, s_in=None, p_in=None,
                nthreads=None):
    """Step-by-step emulation of the fused MX forward.  fmt_p: 0/1/2/4 exp path, 3 EFQ.

    EFQ codes are clamp(rne(fmaf(s, fp32(efq_a c), fp32(beta - fp32(efq_a (M + E))))), 0, 7)
    with the block exponent E = floor(tmax + phi) - 2 (phi applies to EFQ only; the exp
    path keeps the OCP rule).  s_in (float32 [rows, Skp], optional): raw scores to use
    instead of the emulation's own (a kernel's scores); with dump=True the result then
    also holds p_alt, the code at the other end of the hardware exp2's uncertainty.
    p_in (uint8 [rows, Skp], optional): P codes to accumulate instead of the
    emulation's own (a kernel's codes, once checked against p_codes / p_alt); the
    ambiguity bound then leaves out code decisions.

    Returns dict(out, fallbacks, tiles); with dump=True also s/p_codes/p_scales/m_frozen;
    with ambiguity=True also amb [rows, D]: the bound on how far a kernel output may lie
    from `out` through code, block-exponent and fallback decisions that fp32 leaves
    undetermined (inf for a row whose fallback decision is undetermined).
    s_perturb (tests only) scales every raw score by 1 + s_perturb."""
    B, H, Hkv, Sq, _, D = _shape(mx, Sk)
    rows = _rows(rows)
    n = len(rows)
    Skp = (Sk + 31) // 32 * 32
    ntiles = (Sk + 127) // 128
    out = np.zeros((n, D), np.float64)
    fb = np.zeros(n, np.int32)
    tv = np.zeros(n, np.int32)
    res = dict(out=out, fallbacks=fb, tiles=tv)
    d = None
    if dump or ambiguity or s_in is not None or p_in is not None:
        d = FsaDump(None, None, None, None, None, None, None, None)
    if p_in is not None:
        p_in = np.ascontiguousarray(p_in, np.uint8)
        assert p_in.shape == (n, Skp)
        d.p_in = p_in.ctypes.data
    if s_in is not None:
        s_in = np.ascontiguousarray(s_in, np.float32)
        assert s_in.shape == (n, Skp)
        d.s_in = s_in.ctypes.data
    if dump:
        res.update(s=np.zeros((n, Skp), np.float32), p_codes=np.zeros((n, Skp), np.uint8),
                   p_scales=np.zeros((n, Skp // 32), np.uint8), m_frozen=np.zeros((n, ntiles), np.float32))
        d.s, d.p_codes, d.p_scales, d.m_frozen = (res["s"].ctypes.data, res["p_codes"].ctypes.data,
                                                  res["p_scales"].ctypes.data, res["m_frozen"].ctypes.data)
        res["p_alt"] = np.zeros((n, Skp), np.uint8)
        d.p_alt = res["p_alt"].ctypes.data
    if ambiguity:
        res["amb"] = np.zeros((n, D), np.float64)
        d.amb = res["amb"].ctypes.data
    g = _geom(B, H, Hkv, Sq, Sk, D, causal)
    ops = mx.struct()
    opts = FsaOpts(float(delta), int(mufu_mask) & 0xFFFFFFFF, float(beta), float(efq_a), float(phi), float(s_perturb))
    lib().orc_fsa_emulate(ctypes.byref(ops), ctypes.byref(g), ctypes.c_float(scale), ctypes.c_int(fmt_p),
                          ctypes.byref(opts), _p(rows), ctypes.c_int64(n), _p(out), _p(fb), _p(tv),
                          ctypes.byref(d) if d is not None else None, ctypes.c_int(nthreads or nthreads_default()))
    return res


def bf16_emulate(q, k, v, causal, scale, rows, tau=8.0, nthreads=None):
    """Emulation of the exact-softmax BF16 kernel (lazy rescale threshold tau, log2 units)."""
    q = np.ascontiguousarray(q, np.uint16); k = np.ascontiguousarray(k, np.uint16)
    v = np.ascontiguousarray(v, np.uint16)
    B, H, Sq, D = q.shape; Hkv, Sk = k.shape[1], k.shape[2]
    rows = _rows(rows)
    out = np.zeros((len(rows), D), np.float64)
    res = np.zeros(len(rows), np.int32)
    g = _geom(B, H, Hkv, Sq, Sk, D, causal)
    lib().orc_bf16_emulate(_p(q), _p(k), _p(v), ctypes.byref(g), ctypes.c_float(scale), ctypes.c_float(tau),
                           _p(rows), ctypes.c_int64(len(rows)), _p(out), _p(res),
                           ctypes.c_int(nthreads or nthreads_default()))
    return dict(out=out, rescales=res)
