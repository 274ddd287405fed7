"""ctypes binding of libfsa (include/fsa.h).  Argument marshalling only: every
step of the computation runs in the library's CUDA kernels; torch provides
device memory and the current stream.  There is no CPU fallback: without the
compiled library every entry point raises."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

FSA_OK, FSA_ERR_INVALID_ARG, FSA_ERR_UNSUPPORTED_FMT, FSA_ERR_LAUNCH, FSA_ERR_TIMEOUT, FSA_ERR_NO_DEVICE = \
    0, -1, -2, -3, -4, -5
FSA_FMT_E4M3, FSA_FMT_E2M3, FSA_FMT_E2M1, FSA_FMT_E2M1_EFQ, FSA_FMT_E3M2, FSA_FMT_NVFP4 = 0, 1, 2, 3, 4, 5
FSA_MX_ROWS, FSA_MX_COLS_T = 0, 1
FSA_EXP_POLY, FSA_EXP_MUFU, FSA_EXP_SPLIT = 0, 1, 2
FMT_BY_NAME = {"E4M3": 0, "E2M3": 1, "E2M1": 2, "E2M1_EFQ": 3, "E3M2": 4, "NVFP4": 5}


class FsaError(RuntimeError):
    def __init__(self, status, what):
        try:
            msg = status_string(status)
        except Exception:  # library not loadable
            msg = "libfsa unavailable"
        super().__init__(f"{what}: {msg} ({status})")
        self.status = status


class fsa_mx_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("fmt", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("S", ctypes.c_int32),
                ("D", ctypes.c_int32)]


class fsa_debug_dump(ctypes.Structure):
    _fields_ = [("s", ctypes.c_void_p), ("m", ctypes.c_void_p), ("p", ctypes.c_void_p), ("p_scales", ctypes.c_void_p),
                ("row_slot", ctypes.c_void_p)]


class fsa_opts(ctypes.Structure):
    _fields_ = [("delta", ctypes.c_float), ("exp_mode", ctypes.c_int32), ("efq_a", ctypes.c_float),
                ("efq_b", ctypes.c_float), ("efq_phi", ctypes.c_float), ("timeout_ms", ctypes.c_uint32),
                ("row_fallbacks", ctypes.c_void_p), ("inject_stall", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("debug", ctypes.POINTER(fsa_debug_dump))]


class fsa_stats(ctypes.Structure):
    _fields_ = [("fallback_events", ctypes.c_uint64), ("row_tiles", ctypes.c_uint64), ("status", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class fsa_layer(ctypes.Structure):
    _fields_ = [("q", ctypes.POINTER(fsa_mx_tensor)), ("k", ctypes.POINTER(fsa_mx_tensor)),
                ("v", ctypes.POINTER(fsa_mx_tensor)), ("out", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("Sq", ctypes.c_int32),
                ("Sk", ctypes.c_int32), ("D", ctypes.c_int32), ("causal", ctypes.c_int32), ("scale", ctypes.c_float),
                ("fmt_qk", ctypes.c_int32), ("fmt_pv", ctypes.c_int32), ("delta", ctypes.c_float),
                ("stats", ctypes.c_void_p)]


class fsa_host_io(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class fsa_device_io(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("q_mx", ctypes.POINTER(fsa_mx_tensor)), ("k_mx", ctypes.POINTER(fsa_mx_tensor)),
                ("v_mx", ctypes.POINTER(fsa_mx_tensor)), ("out", ctypes.c_void_p)]


FSA_OUT_F32, FSA_OUT_BF16 = 0, 1
STATS_BYTES = 24      # fsa_stats: u64 fallback_events, u64 row_tiles, i32 status, i32 reserved

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libfsa.so (building it in-tree first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libfsa.so not found at {path}")
            L = ctypes.CDLL(path)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            L.fsa_mx_sizes.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
            L.fsa_mx_quantize.argtypes = [vp, i, i, i, i, i, i, ctypes.POINTER(fsa_mx_tensor), vp]
            L.fsa_mx_quantize_qkv.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i] + \
                [ctypes.POINTER(fsa_mx_tensor)] * 3 + [vp]
            L.fsa_attention_fwd.argtypes = [ctypes.POINTER(fsa_mx_tensor)] * 3 + [vp, i, i, i, i, i, i, i, f, i, i, vp]
            L.fsa_attention_fwd_ex.argtypes = [ctypes.POINTER(fsa_mx_tensor)] * 3 + \
                [vp, i, i, i, i, i, i, i, f, i, i, ctypes.POINTER(fsa_opts), vp, vp]
            L.fsa_attention_fwd_layers.argtypes = [ctypes.POINTER(fsa_layer), i, ctypes.POINTER(fsa_opts), vp]
            L.fsa_attention_fwd_qbf16.argtypes = [vp] + [ctypes.POINTER(fsa_mx_tensor)] * 2 + \
                [vp, i, i, i, i, i, i, i, f, i, i, ctypes.POINTER(fsa_opts), vp, vp]
            L.fsa_attention_fwd_host.argtypes = [ctypes.POINTER(fsa_host_io), ctypes.POINTER(fsa_device_io),
                                                 i, i, i, i, i, i, i, f, i, i, ctypes.POINTER(fsa_opts), vp, i, vp]
            L.fsa_tune_delta.argtypes = [ctypes.POINTER(fsa_stats), i, f, f, f, ctypes.POINTER(ctypes.c_float)]
            L.fsa_mma_peak.argtypes = [i, i, i, ctypes.c_longlong, vp, ctypes.POINTER(ctypes.c_double), vp]
            L.fsa_bf16_transpose_v.argtypes = [vp, vp, i, i, i, i, vp]
            L.fsa_attention_fwd_bf16.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, vp]
            L.fsa_default_opts.argtypes = [ctypes.POINTER(fsa_opts)]
            L.fsa_default_opts.restype = None
            L.fsa_status_string.argtypes = [i]
            L.fsa_status_string.restype = ctypes.c_char_p
            for n in ("fsa_mx_sizes", "fsa_mx_quantize", "fsa_mx_quantize_qkv", "fsa_attention_fwd",
                      "fsa_attention_fwd_ex", "fsa_bf16_transpose_v", "fsa_attention_fwd_bf16", "fsa_version",
                      "fsa_attention_fwd_layers", "fsa_tune_delta", "fsa_mma_peak", "fsa_attention_fwd_qbf16",
                      "fsa_attention_fwd_host"):
                getattr(L, n).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return load().fsa_status_string(int(s)).decode()


def _check(status, what):
    if status != FSA_OK:
        raise FsaError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _fmt(f):
    return FMT_BY_NAME[f] if isinstance(f, str) else int(f)


def _need_cuda(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise FsaError(FSA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise FsaError(FSA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise FsaError(FSA_ERR_INVALID_ARG, f"{name} must be {dtype}")


# ----------------------------------------------------------------------------- MX tensors
class MxTensor:
    """Device MX tensor: codes and scales owned by torch, described by fsa_mx_tensor."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor, fmt: int, layout: int, B, H, S, D):
        self.codes, self.scales = codes, scales
        self.fmt, self.layout, self.B, self.H, self.S, self.D = int(fmt), int(layout), B, H, S, D

    def struct(self) -> fsa_mx_tensor:
        return fsa_mx_tensor(self.codes.data_ptr(), self.scales.data_ptr(), self.fmt, self.layout,
                             self.B, self.H, self.S, self.D)


def fsa_mx_sizes(B, H, S, D, layout, fmt):
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().fsa_mx_sizes(B, H, S, D, int(layout), _fmt(fmt), ctypes.byref(cb), ctypes.byref(sb)), "fsa_mx_sizes")
    return cb.value, sb.value


def _check_mx_buffers(m: MxTensor, name: str):
    """codes and scales are contiguous uint8 tensors of at least fsa_mx_sizes bytes
    for the tensor's own shape, layout and format (the kernels write and read that
    many bytes; the C ABI receives bare pointers and cannot check)."""
    for t, part in ((m.codes, "codes"), (m.scales, "scales")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or not t.is_contiguous():
            raise FsaError(FSA_ERR_INVALID_ARG, f"{name}.{part} must be a contiguous uint8 tensor")
    cb, sb = fsa_mx_sizes(m.B, m.H, m.S, m.D, m.layout, m.fmt)
    if m.codes.numel() < cb or m.scales.numel() < sb:
        raise FsaError(FSA_ERR_INVALID_ARG, f"{name}: codes/scales hold {m.codes.numel()}/{m.scales.numel()} bytes, "
                                            f"need {cb}/{sb}")


def _need_mx(m: MxTensor, name: str, device):
    """An MX tensor on the given CUDA device with buffers large enough for it."""
    for t, part in ((m.codes, "codes"), (m.scales, "scales")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise FsaError(FSA_ERR_INVALID_ARG, f"{name}.{part} must be a CUDA tensor")
        if t.device != device:
            raise FsaError(FSA_ERR_INVALID_ARG, f"{name}.{part} is on {t.device}, the call on {device}")
    _check_mx_buffers(m, name)


def empty_mx(B, H, S, D, layout, fmt, device) -> MxTensor:
    cb, sb = fsa_mx_sizes(B, H, S, D, layout, fmt)
    return MxTensor(torch.empty(cb, dtype=torch.uint8, device=device), torch.empty(sb, dtype=torch.uint8, device=device),
                    _fmt(fmt), layout, B, H, S, D)


def fsa_mx_quantize(x: torch.Tensor, layout, fmt, out: MxTensor | None = None, stream=None) -> MxTensor:
    """Quantise x (bf16 [B,H,S,D] on the GPU) into an MX tensor (FSA_MX_ROWS for Q/K, FSA_MX_COLS_T for V)."""
    _need_cuda(x, "x", torch.bfloat16)
    B, H, S, D = x.shape
    fmt = _fmt(fmt)
    if out is None:
        out = empty_mx(B, H, S, D, layout, fmt, x.device)
    else:
        out.fmt, out.layout, out.B, out.H, out.S, out.D = fmt, int(layout), B, H, S, D
        _need_mx(out, "out", x.device)
    st = out.struct()
    _check(load().fsa_mx_quantize(ctypes.c_void_p(x.data_ptr()), B, H, S, D, int(layout), fmt, ctypes.byref(st),
                                  _stream(stream)), "fsa_mx_quantize")
    return out


def fsa_mx_quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, fmt_qk, fmt_v,
                        out: tuple | None = None, stream=None) -> tuple:
    """Q, K (FSA_MX_ROWS, fmt_qk) and V (FSA_MX_COLS_T, fmt_v) of one attention call in one launch."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need_cuda(t, n, torch.bfloat16)
    B, H, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Sk, D) or tuple(v.shape) != (B, Hkv, Sk, D):
        raise FsaError(FSA_ERR_INVALID_ARG, "q, k, v shapes")
    fmt_qk, fmt_v = _fmt(fmt_qk), _fmt(fmt_v)
    if out is None:
        out = (empty_mx(B, H, Sq, D, FSA_MX_ROWS, fmt_qk, q.device),
               empty_mx(B, Hkv, Sk, D, FSA_MX_ROWS, fmt_qk, q.device),
               empty_mx(B, Hkv, Sk, D, FSA_MX_COLS_T, fmt_v, q.device))
    else:
        for o, (h, S, layout, f), n in zip(out, ((H, Sq, FSA_MX_ROWS, fmt_qk), (Hkv, Sk, FSA_MX_ROWS, fmt_qk),
                                                 (Hkv, Sk, FSA_MX_COLS_T, fmt_v)), ("q_out", "k_out", "v_out")):
            o.fmt, o.layout, o.B, o.H, o.S, o.D = f, layout, B, h, S, D
            _need_mx(o, n, q.device)
    sq, sk, sv = (o.struct() for o in out)
    _check(load().fsa_mx_quantize_qkv(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                      ctypes.c_void_p(v.data_ptr()), B, H, Hkv, Sq, Sk, D, fmt_qk, fmt_v,
                                      ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv), _stream(stream)),
           "fsa_mx_quantize_qkv")
    return out


def default_opts() -> fsa_opts:
    o = fsa_opts()
    load().fsa_default_opts(ctypes.byref(o))
    return o


def new_stats(device=None) -> torch.Tensor:
    """Zeroed device buffer for fsa_stats (read it back with read_stats)."""
    return torch.zeros(STATS_BYTES // 8, dtype=torch.int64, device=device or "cuda")


def read_stats(stats: torch.Tensor) -> dict:
    v = stats.cpu()
    st = int(v[2].item() & 0xFFFFFFFF)
    st = st - (1 << 32) if st >= 1 << 31 else st
    return dict(fallback_events=int(v[0].item()), row_tiles=int(v[1].item()), status=st)


def _out_dtype(out_dtype):
    if out_dtype in (None, "f32", torch.float32, FSA_OUT_F32):
        return FSA_OUT_F32, torch.float32
    if out_dtype in ("bf16", torch.bfloat16, FSA_OUT_BF16):
        return FSA_OUT_BF16, torch.bfloat16
    raise FsaError(FSA_ERR_INVALID_ARG, f"out_dtype {out_dtype!r}")


def _opts(delta=None, exp_mode=None, efq_a=None, efq_b=None, efq_phi=None, timeout_ms=0, inject_stall=False,
          schedule=None, out_dtype=FSA_OUT_F32) -> fsa_opts:
    o = default_opts()
    if delta is not None:
        o.delta = float(delta)
    if exp_mode is not None:
        o.exp_mode = int(exp_mode)
    if efq_a is not None:
        o.efq_a = float(efq_a)
    if efq_b is not None:
        o.efq_b = float(efq_b)
    if efq_phi is not None:
        o.efq_phi = float(efq_phi)
    if timeout_ms:
        o.timeout_ms = int(timeout_ms)
    o.inject_stall = int(bool(inject_stall))
    if schedule is not None:
        o.schedule = int(schedule)
    o.out_dtype = int(out_dtype)
    return o


class DebugDump:
    """Device buffers for the debug instance's per-tile dumps (fsa_debug_dump): every
    query row, or only `rows` (global row ids, dumped in that order).  Entries the
    kernel does not write keep their initial values: scores -inf, M NaN, words 0."""

    def __init__(self, B, H, Sq, Sk, device=None, rows=None):
        R, nkt = B * H * Sq, (Sk + 127) // 128
        dev = device or "cuda"
        self.row_slot = None
        if rows is not None:
            rows = torch.as_tensor(rows, dtype=torch.int64)
            slot = torch.full((R,), -1, dtype=torch.int32)
            slot[rows] = torch.arange(len(rows), dtype=torch.int32)
            self.row_slot = slot.to(dev)
            R = len(rows)
        self.n_rows, self.nkt = R, nkt
        self.s = torch.full((R, nkt * 128), float("-inf"), dtype=torch.float32, device=dev)
        self.m = torch.full((R, nkt), float("nan"), dtype=torch.float32, device=dev)
        self.p = torch.zeros((R, nkt, 32), dtype=torch.int32, device=dev)
        self.p_scales = torch.zeros((R, nkt), dtype=torch.int32, device=dev)

    def struct(self) -> fsa_debug_dump:
        return fsa_debug_dump(self.s.data_ptr(), self.m.data_ptr(), self.p.data_ptr(), self.p_scales.data_ptr(),
                              self.row_slot.data_ptr() if self.row_slot is not None else 0)


def fsa_attention_fwd(q, k: MxTensor, v: MxTensor, out: torch.Tensor | None = None, *, Hkv=None,
                      causal=False, scale=None, fmt_qk=None, fmt_pv=None, delta=None, exp_mode=None,
                      efq_a=None, efq_b=None, efq_phi=None, timeout_ms=0,
                      row_fallbacks: torch.Tensor | None = None, stats=None, inject_stall=False, schedule=None,
                      out_dtype=None, debug: DebugDump | None = None, stream=None) -> torch.Tensor:
    """O [B,H,Sq,D] (fp32, or bf16 with out_dtype="bf16") by the fused MX forward.  q is an
    MxTensor (fsa_attention_fwd_ex) or a bf16 [B,H,Sq,D] CUDA tensor, quantised to fmt_qk
    in the kernel's prologue (fsa_attention_fwd_qbf16)."""
    q_raw = isinstance(q, torch.Tensor)
    if q_raw:
        _need_cuda(q, "q", torch.bfloat16)
        B, H, Sq, D = q.shape
        if fmt_qk is None:
            raise FsaError(FSA_ERR_INVALID_ARG, "a bf16 q needs fmt_qk")
    else:
        B, H, Sq, D = q.B, q.H, q.S, q.D
    Hkv = k.H if Hkv is None else Hkv
    Sk = k.S
    scale = D ** -0.5 if scale is None else scale
    fmt_qk = q.fmt if fmt_qk is None else _fmt(fmt_qk)
    fmt_pv = v.fmt if fmt_pv is None else _fmt(fmt_pv)
    od, tdt = _out_dtype(out_dtype if out is None or out_dtype is not None else out.dtype)
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=tdt, device=k.codes.device)
    _need_cuda(out, "out", tdt)
    if out.numel() < B * H * Sq * D:
        raise FsaError(FSA_ERR_INVALID_ARG, "out is smaller than B*H*Sq*D")
    for m, n in (((k, "k"), (v, "v")) if q_raw else ((q, "q"), (k, "k"), (v, "v"))):
        _need_mx(m, n, out.device)
    if q_raw and q.device != out.device:
        raise FsaError(FSA_ERR_INVALID_ARG, f"q is on {q.device}, the call on {out.device}")
    if stats is not None:
        _need_cuda(stats, "stats")
        if stats.device != out.device or stats.numel() * stats.element_size() < STATS_BYTES:
            raise FsaError(FSA_ERR_INVALID_ARG, f"stats must hold {STATS_BYTES} bytes on {out.device}")
    o = _opts(delta, exp_mode, efq_a, efq_b, efq_phi, timeout_ms, inject_stall, schedule, od)
    if row_fallbacks is not None:
        _need_cuda(row_fallbacks, "row_fallbacks", torch.int32)
        if row_fallbacks.device != out.device or row_fallbacks.numel() < B * H * Sq:
            raise FsaError(FSA_ERR_INVALID_ARG, f"row_fallbacks must hold B*H*Sq int32 on {out.device}")
        o.row_fallbacks = row_fallbacks.data_ptr()
    if debug is not None:
        nkt = (Sk + 127) // 128
        nslot = debug.n_rows if debug.row_slot is not None else B * H * Sq
        if debug.nkt != nkt:
            raise FsaError(FSA_ERR_INVALID_ARG, "debug dump made for another key length")
        for t, n, cols in ((debug.s, "s", nkt * 128), (debug.m, "m", nkt), (debug.p, "p", nkt * 32),
                           (debug.p_scales, "p_scales", nkt)):
            _need_cuda(t, f"debug.{n}")
            if t.device != out.device or t.numel() < nslot * cols:
                raise FsaError(FSA_ERR_INVALID_ARG, f"debug.{n} is too small")
        if debug.row_slot is not None and (debug.row_slot.numel() != B * H * Sq or debug.row_slot.device != out.device):
            raise FsaError(FSA_ERR_INVALID_ARG, "debug.row_slot must hold B*H*Sq slots on the output's device")
        dd = debug.struct()
        o.debug = ctypes.pointer(dd)
    ks, vs = k.struct(), v.struct()
    tail = (ctypes.c_void_p(out.data_ptr()), B, H, Hkv, Sq, Sk, D, int(bool(causal)), float(scale), fmt_qk, fmt_pv,
            ctypes.byref(o), ctypes.c_void_p(stats.data_ptr() if stats is not None else 0), _stream(stream))
    if q_raw:
        _check(load().fsa_attention_fwd_qbf16(ctypes.c_void_p(q.data_ptr()), ctypes.byref(ks), ctypes.byref(vs),
                                              *tail), "fsa_attention_fwd_qbf16")
    else:
        qs = q.struct()
        _check(load().fsa_attention_fwd_ex(ctypes.byref(qs), ctypes.byref(ks), ctypes.byref(vs), *tail),
               "fsa_attention_fwd_ex")
    return out


def fsa_attention_fwd_layers(layers, *, out_dtype=None, stream=None, **opt_kw) -> list:
    """Several attention layers, each with its own formats and margin, back to back on one
    stream (fsa_attention_fwd_layers).  layers: dicts with q, k, v (MxTensor), causal,
    scale, fmt_qk, fmt_pv, delta, optional out and stats.  Returns the outputs."""
    od, tdt = _out_dtype(out_dtype)
    n = len(layers)
    arr = (fsa_layer * max(n, 1))()
    keep, outs = [], []
    for i, L in enumerate(layers):
        q, k, v = L["q"], L["k"], L["v"]
        out = L.get("out")
        if out is None:
            out = torch.empty((q.B, q.H, q.S, q.D), dtype=tdt, device=q.codes.device)
        _need_cuda(out, "out", tdt)
        if out.numel() < q.B * q.H * q.S * q.D:
            raise FsaError(FSA_ERR_INVALID_ARG, "out is smaller than B*H*Sq*D")
        for m, nm in ((q, "q"), (k, "k"), (v, "v")):
            _need_mx(m, nm, out.device)
        st = L.get("stats")
        if st is not None:
            _need_cuda(st, "stats")
            if st.device != out.device or st.numel() * st.element_size() < STATS_BYTES:
                raise FsaError(FSA_ERR_INVALID_ARG, f"stats must hold {STATS_BYTES} bytes on {out.device}")
        structs = (q.struct(), k.struct(), v.struct())
        keep.append(structs)
        fq = q.fmt if L.get("fmt_qk") is None else _fmt(L["fmt_qk"])
        fp = v.fmt if L.get("fmt_pv") is None else _fmt(L["fmt_pv"])
        scale = L.get("scale") or q.D ** -0.5
        arr[i] = fsa_layer(ctypes.pointer(structs[0]), ctypes.pointer(structs[1]), ctypes.pointer(structs[2]),
                           out.data_ptr(), q.B, q.H, k.H, q.S, k.S, q.D, int(bool(L.get("causal", False))),
                           float(scale), fq, fp, float(L.get("delta", 8.0)), st.data_ptr() if st is not None else 0)
        outs.append(out)
    o = _opts(out_dtype=od, **opt_kw)
    _check(load().fsa_attention_fwd_layers(arr, n, ctypes.byref(o), _stream(stream)), "fsa_attention_fwd_layers")
    return outs


class HostCallBuffers:
    """Device buffers of fsa_attention_fwd_host for one call shape and format pair:
    bf16 Q, K, V, the three MX tensors and the output, all owned by torch."""

    def __init__(self, B, H, Hkv, Sq, Sk, D, fmt_qk, fmt_pv, out_dtype=None, device=None):
        dev = torch.device(device or "cuda")
        fmt_qk, fmt_pv = _fmt(fmt_qk), _fmt(fmt_pv)
        fv = FSA_FMT_E2M1 if fmt_pv == FSA_FMT_E2M1_EFQ else fmt_pv
        _, tdt = _out_dtype(out_dtype)
        self.shape = (B, H, Hkv, Sq, Sk, D)
        self.q = torch.empty((B, H, Sq, D), dtype=torch.bfloat16, device=dev)
        self.k = torch.empty((B, Hkv, Sk, D), dtype=torch.bfloat16, device=dev)
        self.v = torch.empty((B, Hkv, Sk, D), dtype=torch.bfloat16, device=dev)
        self.mx = (empty_mx(B, H, Sq, D, FSA_MX_ROWS, fmt_qk, dev), empty_mx(B, Hkv, Sk, D, FSA_MX_ROWS, fmt_qk, dev),
                   empty_mx(B, Hkv, Sk, D, FSA_MX_COLS_T, fv, dev))
        self.out = torch.empty((B, H, Sq, D), dtype=tdt, device=dev)

    @classmethod
    def from_tensors(cls, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mx, out: torch.Tensor):
        """Wrap existing device tensors (bf16 q, k, v; the (q, k, v) MxTensors; out)."""
        self = cls.__new__(cls)
        B, H, Sq, D = q.shape
        self.shape = (B, H, k.shape[1], Sq, k.shape[2], D)
        self.q, self.k, self.v, self.mx, self.out = q, k, v, tuple(mx), out
        return self


def fsa_attention_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor | None = None, *,
                           buffers: HostCallBuffers | None = None, fmt_qk="E4M3", fmt_pv="E4M3", causal=False,
                           scale=None, n_chunks=0, stats=None, row_fallbacks: torch.Tensor | None = None,
                           out_dtype=None, stream=None, **opt_kw) -> torch.Tensor:
    """O [B,H,Sq,D] in host memory from bf16 q, k, v in host memory (fsa_attention_fwd_host):
    copies in, quantisation, attention and copies back by groups of kv heads, the copies
    overlapping the compute.  Page-locked (pinned) tensors give the overlap.  The work is
    enqueued on `stream` (default: the current one): synchronise it before reading out."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise FsaError(FSA_ERR_INVALID_ARG, f"{n} must be a contiguous bf16 host tensor")
    B, H, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Sk, D) or tuple(v.shape) != (B, Hkv, Sk, D):
        raise FsaError(FSA_ERR_INVALID_ARG, "q, k, v shapes")
    fmt_qk, fmt_pv = _fmt(fmt_qk), _fmt(fmt_pv)
    od, tdt = _out_dtype(out_dtype if out is None or out_dtype is not None else out.dtype)
    if buffers is None:
        buffers = HostCallBuffers(B, H, Hkv, Sq, Sk, D, fmt_qk, fmt_pv, tdt)
    if buffers.shape != (B, H, Hkv, Sq, Sk, D) or buffers.out.dtype != tdt:
        raise FsaError(FSA_ERR_INVALID_ARG, "buffers were made for another shape or output dtype")
    dev = buffers.out.device
    for t, n in ((buffers.q, "buffers.q"), (buffers.k, "buffers.k"), (buffers.v, "buffers.v"),
                 (buffers.out, "buffers.out")):
        _need_cuda(t, n)
    fv = FSA_FMT_E2M1 if fmt_pv == FSA_FMT_E2M1_EFQ else fmt_pv
    for m, (f, layout), n in zip(buffers.mx, ((fmt_qk, FSA_MX_ROWS), (fmt_qk, FSA_MX_ROWS), (fv, FSA_MX_COLS_T)),
                                 ("q_mx", "k_mx", "v_mx")):
        if m.fmt != f or m.layout != layout:
            raise FsaError(FSA_ERR_INVALID_ARG, f"buffers.{n} was made for another format")
        _need_mx(m, f"buffers.{n}", dev)
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=tdt, pin_memory=True)
    if out.is_cuda or out.dtype != tdt or not out.is_contiguous() or out.numel() < B * H * Sq * D:
        raise FsaError(FSA_ERR_INVALID_ARG, f"out must be a contiguous {tdt} host tensor of B*H*Sq*D elements")
    if stats is not None:
        _need_cuda(stats, "stats")
        if stats.device != dev or stats.numel() * stats.element_size() < STATS_BYTES:
            raise FsaError(FSA_ERR_INVALID_ARG, f"stats must hold {STATS_BYTES} bytes on {dev}")
    o = _opts(out_dtype=od, **opt_kw)
    if row_fallbacks is not None:
        _need_cuda(row_fallbacks, "row_fallbacks", torch.int32)
        if row_fallbacks.device != dev or row_fallbacks.numel() < B * H * Sq:
            raise FsaError(FSA_ERR_INVALID_ARG, f"row_fallbacks must hold B*H*Sq int32 on {dev}")
        o.row_fallbacks = row_fallbacks.data_ptr()
    hio = fsa_host_io(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr())
    structs = tuple(m.struct() for m in buffers.mx)
    dio = fsa_device_io(buffers.q.data_ptr(), buffers.k.data_ptr(), buffers.v.data_ptr(),
                        ctypes.pointer(structs[0]), ctypes.pointer(structs[1]), ctypes.pointer(structs[2]),
                        buffers.out.data_ptr())
    scale = D ** -0.5 if scale is None else scale
    _check(load().fsa_attention_fwd_host(ctypes.byref(hio), ctypes.byref(dio), B, H, Hkv, Sq, Sk, D,
                                         int(bool(causal)), float(scale), fmt_qk, fmt_pv, ctypes.byref(o),
                                         ctypes.c_void_p(stats.data_ptr() if stats is not None else 0),
                                         int(n_chunks), _stream(stream)), "fsa_attention_fwd_host")
    return out


def fsa_tune_delta(stats: list, deltas: list, target_rate=0.01, step=4.0, max_delta=64.0) -> list:
    """Host-side margin update from per-layer stats dicts (read_stats); returns new margins."""
    n = len(stats)
    sarr = (fsa_stats * max(n, 1))()
    for i, st in enumerate(stats):
        sarr[i] = fsa_stats(int(st["fallback_events"]), int(st["row_tiles"]), int(st["status"]), 0)
    d = (ctypes.c_float * max(n, 1))(*[float(x) for x in deltas])
    _check(load().fsa_tune_delta(sarr, n, float(target_rate), float(step), float(max_delta), d), "fsa_tune_delta")
    return [float(d[i]) for i in range(n)]


def fsa_mma_peak(kind: int, n_ctas: int, iters: int, status: torch.Tensor | None = None, n: int = 128,
                 stream=None) -> float:
    """Launch the tensor-core throughput probe (M=128, N=n); returns the launch's FLOPs
    (time it with events)."""
    fl = ctypes.c_double()
    ptr = 0
    if status is not None:
        _need_cuda(status, "status", torch.int32)
        ptr = status.data_ptr()
    _check(load().fsa_mma_peak(int(kind), int(n), int(n_ctas), int(iters), ctypes.c_void_p(ptr), ctypes.byref(fl),
                               _stream(stream)), "fsa_mma_peak")
    return fl.value


def fsa_bf16_transpose_v(v: torch.Tensor, vt: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need_cuda(v, "v", torch.bfloat16)
    B, Hkv, S, D = v.shape
    Sp = (S + 127) // 128 * 128
    if vt is None:
        vt = torch.empty((B, Hkv, D, Sp), dtype=torch.bfloat16, device=v.device)
    _check(load().fsa_bf16_transpose_v(ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(vt.data_ptr()), B, Hkv, S, D,
                                       _stream(stream)), "fsa_bf16_transpose_v")
    return vt


def fsa_attention_fwd_bf16(q: torch.Tensor, k: torch.Tensor, vt: torch.Tensor, out: torch.Tensor | None = None, *,
                           causal=False, scale=None, stats=None, stream=None) -> torch.Tensor:
    """O [B,H,Sq,D] fp32 by the exact-softmax BF16 kernel; vt from fsa_bf16_transpose_v."""
    for t, n in ((q, "q"), (k, "k"), (vt, "vt")):
        _need_cuda(t, n, torch.bfloat16)
    B, H, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    scale = D ** -0.5 if scale is None else scale
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=torch.float32, device=q.device)
    _check(load().fsa_attention_fwd_bf16(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                         ctypes.c_void_p(vt.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                         B, H, Hkv, Sq, Sk, D, int(bool(causal)), float(scale),
                                         ctypes.c_void_p(stats.data_ptr() if stats is not None else 0),
                                         _stream(stream)), "fsa_attention_fwd_bf16")
    return out
