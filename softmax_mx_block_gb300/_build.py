"""In-tree build of libfsa.so (nvcc, sm_103a only).

The fused attention kernel is compiled once per (QK format, PV format) pair in
its own translation unit so that the pairs build in parallel."""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]

# (QK format, PV format): 0 E4M3, 1 E2M3, 2 E2M1, 3 E2M1 by the EFQ rule, 4 E3M2, 5 BF16, 6 NVFP4 (Q/K)
ATTN_PAIRS = [(qk, pv) for qk in (0, 1, 2, 4, 6) for pv in range(5)] + [(5, 5)]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def _units():
    units = [("fsa_api", os.path.join(CSRC, "fsa_api.cu"), []),
             ("fsa_quant", os.path.join(CSRC, "fsa_quant.cu"), []),
             ("fsa_peak", os.path.join(CSRC, "fsa_peak.cu"), [])]
    for qk, pv in ATTN_PAIRS:
        units.append((f"fsa_attn_{qk}{pv}", os.path.join(CSRC, "fsa_attn.cu"),
                      [f"-DFSA_INST_QK={qk}", f"-DFSA_INST_PV={pv}"]))
    return units


def _newest_input() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libfsa.so in the package dir."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    nvcc = _nvcc()

    def compile_unit(u):
        name, src, defs = u
        obj = os.path.join(OBJ, name + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defs, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    jobs = jobs or min(16, os.cpu_count() or 4)
    with ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(compile_unit, _units()))
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
