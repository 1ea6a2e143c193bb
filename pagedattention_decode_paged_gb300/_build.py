"""Compile the CUDA sources into the in-tree shared library libpagedattn.so.

nvcc, one -gencode for sm_103a, translation units compiled in parallel and
linked with -shared.  The output lands in pagedattention_decode_paged_gb300/
_lib/ (git-ignored) so the library that tests and benchmarks load is always
the one built from this tree on this machine.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIBDIR = PKG / "_lib"
LIB = LIBDIR / "libpagedattn.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "append.cu", "decode_simt.cu", "decode_gqa_tc.cu", "decode_balanced_simt.cu",
           "decode_balanced_tc.cu", "decode_int8.cu", "decode_prefix_tc.cu", "reduce.cu",
           "decode_int8_tc.cu", "decode_gqa_umma.cu"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = Path(cuda) / "bin" / "nvcc"
    return str(path) if path.exists() else (shutil.which("nvcc") or "nvcc")


def _flags(verbose_ptxas: bool) -> list[str]:
    flags = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
             f"-I{INCLUDE}", f"-I{CSRC}", "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def _stale() -> bool:
    if not LIB.exists():
        return True
    built = LIB.stat().st_mtime
    inputs = list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        list(INCLUDE.glob("*.h")) + [Path(__file__)]
    return any(p.stat().st_mtime > built for p in inputs)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> Path:
    """Build libpagedattn.so if any source is newer than it; return its path."""
    if not force and not verbose_ptxas and not _stale():
        return LIB
    LIBDIR.mkdir(exist_ok=True)
    nvcc = _nvcc()
    objdir = LIBDIR / "obj"
    objdir.mkdir(exist_ok=True)
    flags = _flags(verbose_ptxas)

    def compile_one(src: str) -> tuple[str, str]:
        obj = objdir / (Path(src).stem + ".o")
        cmd = [nvcc, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return str(obj), res.stderr

    with ThreadPoolExecutor(max_workers=jobs or min(len(SOURCES), os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for src, (_, log) in zip(SOURCES, results):
            sys.stderr.write(f"== {src}\n{log}")
    tmp = LIBDIR / f".libpagedattn.{os.getpid()}.so"
    link = [nvcc, *ARCH, "-shared", "-o", str(tmp), *[o for o, _ in results], "-lcudart"]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
