"""Build libdgattn.so in-tree with nvcc for sm_103a (no cmake; the translation units compile in
parallel, then one link).  ``python -m gqa_canvas_attention_gb300.build`` or ``build()``."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "dgattn")
LIB = os.path.join(PKG, "libdgattn.so")
SOURCES = ["api.cu", "norm_rope.cu", "attn_fp32.cu", "attn_tc.cu", "attn_tc_split.cu",
           "aux_kernels.cu", "noalloc.cu", "proj_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


ATTN_KERNEL_SOURCES = ["attn_tc_kernel.cuh", "attn_tc.cu", "sm103_ptx.cuh", "dg_internal.cuh",
                       "api.cu"]


def attn_kernel_source_id() -> str:
    """sha1 over the files that fix the tensor-core attention kernel and its launch (the kernel,
    its PTX wrappers, the shared parameter blocks, the launch and schedule code): DRAM counters
    taken from an ncu capture stand for the kernel only while this id is unchanged."""
    import hashlib
    h = hashlib.sha1()
    for name in ATTN_KERNEL_SOURCES:
        h.update(name.encode())
        with open(os.path.join(CSRC, name), "rb") as fh:
            h.update(fh.read())
    return "sha1:" + h.hexdigest()


def source_id() -> str:
    """sha1 over the CUDA sources and the C header the library is built from (file names and
    contents, in name order): the string libdgattn.so reports through dg_attn_build_id()."""
    import hashlib
    h = hashlib.sha1()
    files = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))
    for name, path in [(f, os.path.join(CSRC, f)) for f in files] + \
            [("dg_attn.h", os.path.join(INCLUDE, "dg_attn.h"))]:
        h.update(name.encode())
        with open(path, "rb") as fh:
            h.update(fh.read())
    return "sha1:" + h.hexdigest()


def _flags(verbose_ptxas: bool) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "--expt-relaxed-constexpr", f'-DDG_BUILD_ID="{source_id()}"']
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(outputs: str, inputs: list) -> bool:
    if not os.path.exists(outputs):
        return True
    t = os.path.getmtime(outputs)
    return any(os.path.getmtime(i) > t for i in inputs)


def _built_id():
    """The build id of the library on disk, read without loading it into this process (the
    binding caches the first library it loads), or None."""
    if not os.path.exists(LIB):
        return None
    with open(LIB, "rb") as f:
        data = f.read()
    i = data.find(b"sha1:")
    if i < 0:
        return None
    j = data.find(b"\0", i)
    return data[i:j].decode(errors="replace")


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile every .cu under csrc/ and link libdgattn.so next to this file; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dg_attn.h")]
    if not force and not verbose_ptxas and not _stale(LIB, deps) and _built_id() == source_id():
        return LIB
    nvcc = _nvcc()
    flags = _flags(verbose_ptxas)

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose_ptxas:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
