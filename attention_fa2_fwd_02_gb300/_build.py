"""Build step for libfa.so: nvcc for sm_103a, in-tree, no cmake.

The translation units compile in parallel (one -gencode, sm_103a only) and
are linked into ``attention_fa2_fwd_02_gb300/_build/libfa.so``.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT_DIR = PKG / "_build"
LIB = OUT_DIR / "libfa.so"
SOURCES = ["fa_api.cu", "fa_tc_bf16.cu", "fa_tc_bf16_split.cu",
           "fa_noalloc.cu", "fa_bwd.cu",
           "fa_tc_bf16_varlen.cu", "fa_tc_wide.cu", "fa_tc_wide_fp32.cu",
           "fa_tc_wide_fp32_vt.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    cand = Path("/usr/local/cuda/bin/nvcc")
    return str(cand) if cand.exists() else "nvcc"


def _flags(ptxas_verbose: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", str(INCLUDE), "-I", str(CSRC)]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _inputs() -> list[Path]:
    return sorted(CSRC.glob("*.cu")) + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + \
        sorted(INCLUDE.glob("*.h")) + [Path(__file__)]


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> Path:
    """Compile every CUDA source for sm_103a and link libfa.so; returns its path."""
    if not force and not ptxas_verbose and up_to_date():
        return LIB
    OUT_DIR.mkdir(parents=True, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags(ptxas_verbose)

    def compile_one(src: str) -> tuple[str, str]:
        obj = OUT_DIR / (Path(src).stem + ".o")
        cmd = [nvcc, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return str(obj), r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if not quiet:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = OUT_DIR / f"libfa.so.tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *[o for o, _ in results], "-lcuda"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
