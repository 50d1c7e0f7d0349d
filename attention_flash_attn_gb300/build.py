"""Builds libattn_gb300.so in-tree from csrc/*.cu with nvcc for sm_103a.

Every translation unit is compiled in parallel (one nvcc process each) into ``_build/``
and linked into ``attention_flash_attn_gb300/libattn_gb300.so`` with the CUDA runtime
linked statically, so the library loads without a GPU or a driver (the driver entry
points it needs are resolved at run time).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libattn_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stamp() -> str:
    h = hashlib.sha256()
    files = _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")))
    files.append(os.path.join(ROOT, "include", "attn_gb300.h"))
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())  # relative: the same sources hash alike anywhere
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


# Sources that the backward main kernel's code depends on: a DRAM-traffic figure recorded by
# ncu for that kernel stays valid while these files (and the flags) are unchanged.
BWD_MAIN_SOURCES = ("bwd_tc.cu", "bwd_score.cuh", "tc_common.cuh", "tc_host.cu", "common.cuh", "internal.h")


def _code_only(text: str) -> str:
    """C / C++ source with comments and whitespace removed (string literals kept), so that an
    edit to comments alone leaves a kernel's stamp unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_stamp(names=BWD_MAIN_SOURCES) -> str:
    """Hash of the code (comments and whitespace removed) of the named csrc files and the
    public header, and of the compile flags."""
    h = hashlib.sha256()
    files = [os.path.join(CSRC, n) for n in names] + [os.path.join(ROOT, "include", "attn_gb300.h")]
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the path of the shared library."""
    os.makedirs(BUILD, exist_ok=True)
    stamp_file = os.path.join(BUILD, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        if open(stamp_file).read() == stamp:
            return LIB
    nvcc = _nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    log = "\n".join(err for _, err in results)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as fh:
        fh.write(log)
    if verbose:
        print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "--cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
