"""Scan of the EFQ direct-code rule on the long-context workload, oracle only.

The EFQ-Softmax page (abstract) maps shifted scores, per 32-key block, to a
"normalized residual domain" under an exponent-only scale taken from the local
maximum, then to nonnegative E2M1 codes by "a single affine rule"; it prints no
constants.  This script measures, for each rule of that family,

    E    = clamp(floor(fp32(tmax + phi)) - 2, -127, 127)     (block scale exponent)
    y    = fmaf(s, fp32(a c), fp32(b - fp32(a (M + E))))     (a * residual + b, one FMA)
    code = clamp(rne(y), 0, 7)                               (E2M1 code)

the error of the emulated attention output against fp64 exact attention, as a
multiple of the error floor: exact softmax with the same MX operands, P rounded
to E2M1 (nearest, ties to even) under the OCP scale rule (the floor of the
Fused-Softmax brief, abstract).  The first reading of the rule was a = b = 2,
phi = 0 (the E2M1 code index as twice the log2 of its value, plus 2); the kernels
and the oracle use the constants this scan selects (oracle.EFQ_A, EFQ_B, EFQ_PHI).

Inputs: the long-context workload (B1 H32 Hkv8 D128 causal, N(0,1) Q/K/V in
bf16, MXFP4 QK^T and V) from workloads.py, on seeded sampled query rows.

    python oracle/efq_scan.py [--seq 16384] [--per-head 32] [--grid coarse|fine]

Calls only oracle/ and workloads.py; prints one line per rule and the best rule.
"""
from __future__ import annotations

import argparse
import itertools
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import WORKLOADS, generate, sample_rows  # noqa: E402


def rel_err(a, ref):
    return float(np.linalg.norm(a - ref) / np.linalg.norm(ref))


def grid(kind):
    if kind == "coarse":
        a = [1.5, 1.75, 2.0, 2.25, 2.5]
        b = [1.0, 1.5, 2.0, 2.5, 3.0, 3.5]
        phi = [0.0, 0.25, 0.5, 0.75]
    elif kind == "fine":
        a = [1.6, 1.65, 1.7, 1.75, 1.8, 1.85, 1.9]
        b = [3.0, 3.25, 3.5, 3.75, 4.0, 4.25]
        phi = [0.375, 0.5, 0.625]
    else:
        a = [1.625, 1.6875, 1.75]
        b = [3.25, 3.375, 3.5, 3.625, 3.75]
        phi = [0.4375, 0.5, 0.5625]
    return list(itertools.product(a, b, phi))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--seq", type=int, default=16384, choices=[16384, 32768, 65536, 131072])
    ap.add_argument("--per-head", type=int, default=32)
    ap.add_argument("--grid", default="coarse", choices=["coarse", "fine", "focus", "default"])
    ap.add_argument("--rule", action="append", default=[], help="extra rule a,b,phi")
    ap.add_argument("--row-seed", type=int, default=7777, help="seed offset of the sampled rows")
    args = ap.parse_args()
    w = WORKLOADS[f"long_efq_{args.seq // 1024}k"]
    t0 = time.time()
    q, k, v = generate(w)
    rows = sample_rows(w, per_head=args.per_head, seed_offset=args.row_seed)
    mx = oracle.MxInputs.from_bf16(q, k, v, 2, 2)
    exact = oracle.attn_exact(q, k, v, w.causal, w.scale, rows)
    floor = oracle.attn_floor(mx, w.Sk, w.causal, w.scale, 2, rows)
    e_floor = rel_err(floor, exact)
    exp_path = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, 2, rows, delta=8.0, mufu_mask=0xFFFFFFFF)["out"]
    print(f"# {w.name}: {len(rows)} sampled rows, setup {time.time() - t0:.1f} s; floor error {e_floor:.5f}; "
          f"exp-then-round path {rel_err(exp_path, exact) / e_floor:.3f}x floor", flush=True)
    rules = [(2.0, 2.0, 0.0)] + ([] if args.grid == "default" else grid(args.grid))
    rules += [tuple(float(x) for x in r.split(",")) for r in args.rule]
    print("# a      b      phi    error/floor", flush=True)
    best = None
    for a, b, phi in rules:
        out = oracle.fsa_emulate(mx, w.Sk, w.causal, w.scale, 3, rows, delta=8.0, beta=b, efq_a=a, phi=phi)["out"]
        ratio = rel_err(out, exact) / e_floor
        print(f"{a:6.3f} {b:6.3f} {phi:6.3f} {ratio:8.4f}", flush=True)
        if best is None or ratio < best[0]:
            best = (ratio, a, b, phi)
    print(f"# best: a={best[1]} b={best[2]} phi={best[3]}: {best[0]:.4f}x floor", flush=True)


if __name__ == "__main__":
    main()
