"""Builds the CUDA library libtd.so in-tree (``decode_attention_split_gb300/_build``).

One ``-gencode arch=compute_103a,code=sm_103a`` target (GB300), translation units compiled
in parallel, the CUDA runtime linked statically with its symbols kept private. ptxas
resource usage (registers, spills, shared memory) is kept in ``_build/ptxas.log``.
Run ``python -m decode_attention_split_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libtd.so")
PTXAS_LOG = os.path.join(BUILD, "ptxas.log")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libtd)")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src: str, obj: str, extra: list[str]) -> str:
    cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
           f"-I{INCLUDE}", f"-I{CSRC}", *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}\n{r.stdout}")
    return f"== {os.path.basename(src)}\n{r.stderr}"


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile every .cu under csrc/ and link libtd.so; returns its path."""
    if not force and not extra_flags and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    tmpdir = tempfile.mkdtemp(prefix="obj_", dir=BUILD)
    try:
        srcs = sources()
        objs = [os.path.join(tmpdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
            logs = list(ex.map(lambda so: _compile(so[0], so[1], extra_flags or []), zip(srcs, objs)))
        fd, tmp_lib = tempfile.mkstemp(suffix=".so", dir=BUILD)
        os.close(fd)
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--exclude-libs=ALL", *objs, "-o", tmp_lib]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            if os.path.exists(tmp_lib):
                os.unlink(tmp_lib)
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp_lib, LIB)
        with open(PTXAS_LOG, "w") as f:
            f.write("\n".join(logs))
        if verbose:
            print("\n".join(logs))
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
