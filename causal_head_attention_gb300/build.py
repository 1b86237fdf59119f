"""Build librca_attn.so in-tree with nvcc for sm_103a (no torch, no cmake).

Usage: python -m causal_head_attention_gb300.build   (or build() from Python)
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "librca_attn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librca_attn.so")


def sources():
    return sorted(
        os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))
    ) + [os.path.join(INCLUDE, "rca_attn.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in sources())


UNITS = ("rca_attn.cu", "decode.cu", "materialized.cu")  # translation units, compiled in parallel


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    return subprocess.run(cmd, capture_output=True, text=True)


def build(force: bool = False, verbose: bool = False, extra: tuple = ()) -> str:
    if not force and up_to_date():
        return LIB
    from concurrent.futures import ThreadPoolExecutor

    nvcc = nvcc_path()
    # Hidden visibility: only the calls include/rca_attn.h marks RCA_API are exported.
    common = [nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              f"-I{INCLUDE}", *extra]
    objs = [os.path.join(PKG, u[:-3] + ".o") for u in UNITS]
    cmds = [common + ["-c", "-o", o, os.path.join(CSRC, u)] for u, o in zip(UNITS, objs)]
    with ThreadPoolExecutor(len(cmds)) as ex:
        results = list(ex.map(lambda c: _run(c, verbose), cmds))
    for r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    r = _run([nvcc, ARCH, "-shared", "-o", LIB + ".tmp", *objs], verbose)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    for o in objs:
        os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
