"""Build the CUDA library in-tree: nvcc, sm_103a only, one shared object.

    epilogue_chains_gb300/_build/libfusechain.so

Translation units compile in parallel (``-Xptxas -v`` output is kept per unit under
``_build/ptxas/`` for the register/spill report) and are linked with the static CUDA runtime, so
the library loads without a GPU or driver (the C-ABI symbol check runs on CPU-only hosts).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libfusechain.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-Xptxas", "-v", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str) -> str:
    obj = os.path.join(OUT, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    os.makedirs(os.path.join(OUT, "ptxas"), exist_ok=True)
    with open(os.path.join(OUT, "ptxas", os.path.basename(src) + ".log"), "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr[-6000:]}")
    return obj


def build(force: bool = False, jobs: int | None = None) -> str:
    """Compile every translation unit under csrc/ and link libfusechain.so (no-op if current)."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


_FN_RE = re.compile(r"Compiling entry function '([^']+)' for 'sm_103a'")
_SPILL_RE = re.compile(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads")
_REG_RE = re.compile(r"Used (\d+) registers")


def ptxas_report() -> list[dict]:
    """Per kernel (mangled name): registers and spill bytes as printed by ptxas -v."""
    rows = []
    for log in sorted(glob.glob(os.path.join(OUT, "ptxas", "*.log"))):
        cur = None
        with open(log) as f:
            for line in f:
                m = _FN_RE.search(line)
                if m:
                    cur = {"unit": os.path.basename(log)[:-4], "kernel": m.group(1)}
                    rows.append(cur)
                    continue
                if cur is None:
                    continue
                m = _SPILL_RE.search(line)
                if m:
                    cur.update(stack=int(m.group(1)), spill_stores=int(m.group(2)),
                               spill_loads=int(m.group(3)))
                m = _REG_RE.search(line)
                if m:
                    cur["registers"] = int(m.group(1))
    return rows


if __name__ == "__main__":
    print(build(force=True))
