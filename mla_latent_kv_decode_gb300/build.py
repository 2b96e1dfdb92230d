"""Build libmla.so (the C-ABI library) and libmla_synth.so (the input generator's device twin)
in-tree with nvcc for sm_103a.  Translation units compile in parallel; no cmake."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")

LIBMLA_SOURCES = ["mla_api.cu", "append.cu", "combine.cu", "decode_tc.cu", "decode_gather.cu", "decode_shared.cu",
                  "indexer.cu", "proj.cu"]
SYNTH_SOURCES = ["synth.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra: list[str], verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "mla.h"))
    if _newer(obj, [src] + headers):
        cmd = [_nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr.strip():
            print(r.stderr, file=sys.stderr)
    return obj


def _link(objs: list[str], out: str, verbose: bool) -> None:
    if not _newer(out, objs):
        return
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed for {out}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(verbose: bool = False, ptxas_verbose: bool = False) -> list[str]:
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    srcs = [os.path.join(CSRC, s) for s in LIBMLA_SOURCES + SYNTH_SOURCES]
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), srcs))
    lib = os.path.join(PKG, "libmla.so")
    synth = os.path.join(PKG, "libmla_synth.so")
    _link(objs[:len(LIBMLA_SOURCES)], lib, verbose)
    _link(objs[len(LIBMLA_SOURCES):], synth, verbose)
    return [lib, synth]


if __name__ == "__main__":
    print("\n".join(build(verbose=True, ptxas_verbose="-v" in sys.argv)))
