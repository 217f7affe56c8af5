"""Build libmoe.so (the C-ABI MoE layer library) in-tree for sm_103a.

Each .cu under csrc/ is compiled in parallel with nvcc, then linked into
int4_routed_expert_gb300/libmoe.so against the shared CUDA runtime.  The
router translation unit is compiled with contraction off: its arithmetic is
fixed operation by operation.

    python -m int4_routed_expert_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INC = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# per-file extra flags
EXTRA = {"router.cu": ["-fmad=false"]}


def _nvcc() -> str:
    cand = [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]
    for c in cand:
        p = os.path.join(c, "bin", "nvcc") if c else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INC, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", INC, "--expt-relaxed-constexpr"]
    if verbose:
        common += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in _sources():
        name = os.path.basename(src)
        obj = os.path.join(OUT_DIR, name + ".o")
        cmd = [nvcc, "-c", src, "-o", obj] + common + EXTRA.get(name, [])
        procs.append((name, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for name, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((name, text))
        elif verbose and text.strip():
            print(f"--- {name}\n{text}")
    if failed:
        msg = "\n".join(f"--- {n}\n{t}" for n, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc] + ARCH + ["-shared", "--cudart", "shared", "-o", tmp] + objs,
                   check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
