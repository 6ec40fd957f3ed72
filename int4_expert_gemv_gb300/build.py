"""In-tree build of the sm_103a libraries with nvcc (no cmake, no torch JIT).

Produces, next to this file:
  libmoe.so        the C-ABI library (include/moe.h): every kernel of the path
  libmoe_synth.so  the GPU twin of the seeded input generator (data only)
Translation units compile in parallel; cudart is linked statically so the
libraries load on a machine without a GPU (the ABI's validation still runs).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]

LIBS = {
    "libmoe.so": ["abi.cu", "pack.cu", "ffn.cu", "grouped.cu", "head_route.cu", "noalloc.cu",
                  "step.cu", "chain.cu", "lora_merge.cu", "gather.cu"],
    "libmoe_synth.so": ["synth.cu"],
}


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _deps(src: str) -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return [src] + hdrs + [os.path.join(INCLUDE, "moe.h")]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if not _stale(obj, _deps(src)):
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj + ".tmp"]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        with open(os.path.join(BUILD, os.path.basename(src) + ".ptxas.txt"), "w") as f:
            f.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> dict:
    """Compile every library; returns {name: path}.  Rebuilds only stale parts."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    srcs = sorted({s for v in LIBS.values() for s in v})
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = dict(zip(srcs, ex.map(lambda s: _compile(os.path.join(CSRC, s), verbose_ptxas), srcs)))
    out = {}
    for lib, parts in LIBS.items():
        target = os.path.join(PKG, lib)
        deps = [objs[p] for p in parts]
        if force or _stale(target, deps):
            tmp = target + f".tmp{os.getpid()}"
            cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *deps, "-cudart", "static"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed for {lib}:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, target)
        out[lib] = target
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
