"""In-tree build of libjfa.so for sm_103a (nvcc, no cmake).

Each translation unit compiles in its own process; the objects link into
``jagged_sequence_attention_gb300/libjfa.so`` with the CUDA runtime linked
statically, so the library loads on a machine without a GPU driver (tests that
only need the host planner) and only needs the driver when a CUDA call runs.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libjfa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "plan.cpp", "fwd.cu", "fwd_short.cu", "fwd_pack.cu", "bwd.cu", "bwd_dq.cu", "bwd_fused.cu", "bwd_short.cu", "f32.cu", "static_scratch.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return (["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
            + ARCH + list(extra))


def _digest(extra) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "jfa.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(_flags(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of libjfa.so."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "libjfa.stamp")
    dig = _digest(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == dig:
                return LIB
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + _flags(extra_flags) + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-x", "c++"] + cmd[1:]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {src}\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for _, err in results:
            if err:
                print(err, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(dig)
    return LIB


def build_variant(name: str, defines, sources=("fwd.cu",), verbose: bool = False) -> str:
    """A test build of the library: `sources` compiled again with the extra -D `defines`,
    linked with the main build's objects for the other sources, as _build/lib<name>.so.
    Returns its path.  The main library is built first if needed."""
    build()
    out_dir = os.path.join(BUILD, name)
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(BUILD, f"lib{name}.so")
    extra = [f"-D{d}" for d in defines]
    stamp = os.path.join(out_dir, "stamp")
    dig = _digest(extra) + ",".join(sources)
    if os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == dig:
                return lib
    nvcc = _nvcc()
    objs = []
    for src in SOURCES:
        base = os.path.splitext(src)[0] + ".o"
        if src in sources:
            obj = os.path.join(out_dir, base)
            cmd = [nvcc] + _flags(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"compile failed: {src}\n{r.stdout}\n{r.stderr}")
            objs.append(obj)
        else:
            objs.append(os.path.join(BUILD, base))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"], capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(dig)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force=True, extra_flags=extra, verbose=v))
