"""Seeded synthetic inputs for MX attention: shapes, value distributions, seeds.

This module holds no arithmetic of the method (no quantisation, no softmax):
only the workload definitions and numpy random draws, rounded to bf16.  It is
the one module both the CUDA-path tests/bench and the oracle tests import.

Workloads follow the shapes and structures the Fused-Softmax brief (abstract:
MXFP8/6/4 attention kernels, a Wan2.2 video model with a hybrid MXFP6/4
schedule) and the EFQ-Softmax page (abstract: direct E2M1 probability codes,
16K-128K sequence lengths) describe; no public dataset is involved.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

BN = 128          # key tile of the forward kernel (frozen-max granularity)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    fmt_qk: str          # "E4M3" | "E2M3" | "E2M1"
    fmt_pv: str          # "E4M3" | "E2M3" | "E2M1" | "E2M1_EFQ"
    seed: int
    kind: str = "normal"  # "normal" | "k_outliers" | "rank4" | "planted"
    layers: int = 1
    layer_fmts: tuple = field(default_factory=tuple)   # per layer (fmt_qk, fmt_pv) if layers > 1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H*Sq*Sk*D per layer, halved for causal; summed over layers."""
        f = 4.0 * self.B * self.H * self.Sq * self.Sk * self.D
        return (f / 2 if self.causal else f) * self.layers

    def layer(self, l: int) -> "Workload":
        """The single-layer workload of layer l (its formats and seed)."""
        if self.layers == 1:
            return self
        fq, fp = self.layer_fmts[l]
        return replace(self, name=f"{self.name}.L{l}", fmt_qk=fq, fmt_pv=fp, seed=self.seed + l, layers=1,
                       layer_fmts=())


def _long(S, fmt_qk, fmt_pv, tag):
    return Workload(f"long_{tag}_{S // 1024}k", 1, 32, 8, S, S, 128, True, fmt_qk, fmt_pv, 3)


WORKLOADS = {
    # 1. tiny MXFP8 check: every row checked in full
    "tiny": Workload("tiny", 1, 1, 1, 128, 128, 64, False, "E4M3", "E4M3", 0),
    # 2. LLM prefill, GQA 32/8, causal, K with 4 outlier channels per kv head
    "prefill": Workload("prefill", 1, 32, 8, 4096, 4096, 128, True, "E4M3", "E4M3", 1, "k_outliers"),
    # 3. video DiT self-attention over 21x45x80 latent tokens, peaked rows
    "video_dit": Workload("video_dit", 1, 40, 40, 75600, 75600, 128, False, "E2M3", "E2M1", 2, "rank4"),
    # 5. adversarial speculative max, 12 layers alternating MXFP6 / MXFP4
    "adversarial": Workload("adversarial", 2, 24, 24, 8192, 8192, 128, False, "E2M3", "E2M3", 100, "planted",
                            layers=12, layer_fmts=tuple(("E2M3", "E2M3") if l % 2 == 0 else ("E2M1", "E2M1")
                                                        for l in range(12))),
}
# 4. long context with direct E2M1 probability codes, and 4'. the MXFP8 run at the same shapes
for _S in (16384, 32768, 65536, 131072):
    WORKLOADS[f"long_efq_{_S // 1024}k"] = _long(_S, "E2M1", "E2M1_EFQ", "efq")
    WORKLOADS[f"long_fp8_{_S // 1024}k"] = _long(_S, "E4M3", "E4M3", "fp8")
# 4''. the long-context EFQ run with NVFP4 Q and K (16-element E4M3 scales), an
# operand format adjacent to the pages' MX ones
for _S in (16384, 131072):
    WORKLOADS[f"long_nvfp4_{_S // 1024}k"] = _long(_S, "NVFP4", "E2M1_EFQ", "nvfp4")


def small(w: Workload, Sq: int, Sk: int | None = None, H: int | None = None, Hkv: int | None = None,
          B: int | None = None) -> Workload:
    """Same structure and formats at a smaller size (for parity cases the oracle finishes quickly)."""
    Sk = Sq if Sk is None else Sk
    H = w.H if H is None else H
    Hkv = (w.Hkv if w.Hkv <= H else H) if Hkv is None else Hkv
    return replace(w, name=f"{w.name}_small", Sq=Sq, Sk=Sk, H=H, Hkv=Hkv, B=w.B if B is None else B)


# --------------------------------------------------------------------------- bf16 rounding
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (inputs finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, chunk=1 << 24):
    out = np.empty(shape, np.float32)
    flat = out.reshape(-1)
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        flat[s:s + n] = rng.standard_normal(n, dtype=np.float32)
    return out


# --------------------------------------------------------------------------- generators
def generate(w: Workload, layer: int = 0):
    """Q [B,H,Sq,D], K/V [B,Hkv,Sk,D] as bf16 bit patterns (uint16), drawn with
    numpy default_rng(seed) in the order Q, K, V (+ structure draws after)."""
    if w.layers > 1:
        w = w.layer(layer)
    rng = np.random.default_rng(w.seed)
    q = _normal(rng, (w.B, w.H, w.Sq, w.D))
    k = _normal(rng, (w.B, w.Hkv, w.Sk, w.D))
    v = _normal(rng, (w.B, w.Hkv, w.Sk, w.D))
    if w.kind == "k_outliers":
        # 4 channels per kv head, fixed over positions, scaled x8
        for b in range(w.B):
            for h in range(w.Hkv):
                ch = rng.choice(w.D, 4, replace=False)
                k[b, h][:, ch] *= 8.0
    elif w.kind == "rank4":
        # Q, K = 0.5 N(0,1) + a R: R a shared seeded orthonormal 4 x D basis times g,
        # a ~ N(0, I4) per token; g = 4.75 makes the rank-4 score term (times the
        # softmax scale) have std ~4, i.e. peaked rows.
        g = 4.75
        basis, _ = np.linalg.qr(rng.standard_normal((w.D, 4)))
        R = (basis.T * g).astype(np.float32)                      # [4, D]
        q *= 0.5
        k *= 0.5
        for t, S in ((q, w.Sq), (k, w.Sk)):
            for b in range(t.shape[0]):
                for h in range(t.shape[1]):
                    a = rng.standard_normal((S, 4), dtype=np.float32)
                    t[b, h] += a @ R
    elif w.kind == "planted":
        # 1% of keys per (b, h), at positions in [BN, Sk) (never the first tile),
        # set to 6*sqrt(D)*q_i/|q_i| for a random query i: late tiles exceed the frozen max.
        npl = int(round(0.01 * w.Sk))
        for b in range(w.B):
            for h in range(w.Hkv):
                pos = rng.choice(np.arange(BN, w.Sk), npl, replace=False)
                qi = rng.integers(0, w.Sq, npl)
                qq = q[b, h * (w.H // w.Hkv)][qi]
                k[b, h][pos] = 6.0 * math.sqrt(w.D) * qq / np.linalg.norm(qq, axis=1, keepdims=True)
    elif w.kind != "normal":
        raise ValueError(w.kind)
    return to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)


def sample_rows(w: Workload, per_head: int = 256, seed_offset: int = 7777) -> np.ndarray:
    """Query row ids ((b*H + h)*Sq + i): all rows if Sq <= per_head, else per (b, h)
    `per_head` rows drawn without replacement by default_rng(seed + 7777)."""
    if w.Sq <= per_head:
        return np.arange(w.B * w.H * w.Sq, dtype=np.int64)
    rng = np.random.default_rng(w.seed + seed_offset)
    rows = []
    for bh in range(w.B * w.H):
        rows.append(bh * w.Sq + np.sort(rng.choice(w.Sq, per_head, replace=False)))
    return np.concatenate(rows).astype(np.int64)
