"""Builds libcpattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

    python -m context_attention_dits_gb300.build [--verbose-ptxas]

Translation units compile in parallel; the shared library links the CUDA
runtime statically and fetches the one driver entry point it needs
(cuTensorMapEncodeTiled) at run time, so it loads on machines without a GPU
driver.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libcpattn.so")
SOURCES = ["attn_tc.cu", "attn_bwd.cu", "attn_bwd_tc.cu", "kernels_simt.cu", "cp_api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, p.stdout


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    nvcc = nvcc_path()
    build_dir = os.path.join(PKG, "_build")
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "cp_attn.h")]
    newest = max(os.path.getmtime(d) for d in deps)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest and not verbose_ptxas:
        return LIB
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
              "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmds.append(common + ["-c", os.path.join(CSRC, src), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        results = list(ex.map(_run, cmds))
    log = "\n".join(out for _, out in results)
    if any(rc != 0 for rc, _ in results):
        raise RuntimeError("nvcc failed:\n" + log)
    if verbose_ptxas:
        print(log)
    tmp = LIB + ".tmp"
    rc, out = _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
    if rc != 0:
        raise RuntimeError("link failed:\n" + out)
    os.replace(tmp, LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args(argv)
    print(build(verbose_ptxas=args.verbose_ptxas, force=args.force))


if __name__ == "__main__":
    sys.exit(main())
