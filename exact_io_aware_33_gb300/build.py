"""Builds libfa.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under ``csrc/`` is compiled in parallel into
``_build/`` at the repository root and linked into ``libfa.so`` next to this
file. A unit is recompiled only when it, or a header it may include, is
newer than its object file.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfa.so")

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is needed to build libfa.so")


def _headers():
    out = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh")):
                out.append(os.path.join(d, f))
    return out


def build(verbose: bool = False, force: bool = False, extra_flags=None, out_dir: str | None = None,
          lib_path: str | None = None) -> str:
    """Compile the CUDA sources and link libfa.so; returns the library path.

    ``out_dir`` / ``lib_path`` place the objects and the library elsewhere
    (used for test-only variants built with extra ``-D`` flags; the product
    library is always ``libfa.so`` next to this file)."""
    build_dir = out_dir or BUILD
    lib = lib_path or LIB
    os.makedirs(build_dir, exist_ok=True)
    exe = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    newest_header = max(os.path.getmtime(h) for h in _headers())
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(path), newest_header)):
            continue
        cmd = [exe, "-c", path, "-o", obj] + flags
        if verbose:
            cmd.append("-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    if force or procs or not os.path.exists(lib) or any(
            os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        cmd = [exe, "-shared", "-o", tmp] + objs + ARCH
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, lib)
    return lib


# Test-only variant for the bounded-wait (timeout) path: the forward's TMA
# producer never loads the last V tile of its key stream, and every wait gives
# up after 20 ms instead of about a second. It lives under _build/ and is
# never loaded by the package; only tests/test_timeout_path.py uses it.
TIMEOUT_TEST_DIR = os.path.join(BUILD, "timeout_test")
TIMEOUT_TEST_FLAGS = ["-DFA_TEST_SKIP_ARRIVE", "-DFA_WAIT_BUDGET_NS=20000000ull"]


def build_timeout_test_variant(verbose: bool = False) -> str:
    """Build the test-only timeout variant of the library; returns its path."""
    return build(verbose=verbose, extra_flags=TIMEOUT_TEST_FLAGS, out_dir=TIMEOUT_TEST_DIR,
                 lib_path=os.path.join(TIMEOUT_TEST_DIR, "libfa_timeout_test.so"))


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
