"""Build step for the CUDA library ``libgemm_tn.so`` (sm_103a only).

Each translation unit under ``csrc/`` is compiled by nvcc in parallel with one
``-gencode arch=compute_103a,code=sm_103a`` and linked into a shared object in
this package directory. Objects go to ``_build/`` at the repository root.
The CUDA runtime is linked statically, so the library only needs the driver.

    python -m dense_tiled_gemm_03_gb300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import argparse
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
BUILD_DIR = ROOT / "_build" / "gemm_tn"
LIBRARY = PKG / "libgemm_tn.so"

SOURCES = ["gemm_tn_api.cu", "sm103_gemm_1cta.cu", "sm103_gemm_2cta.cu", "sm103_gemm_nn.cu", "sm103_gemm_fused.cu",
           "sm103_flash_attn.cu", "repack.cu", "sm103_gemm_splitk.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", str(INCLUDE), "-I", str(CSRC)]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm_tn.so")
    return cand


def _inputs() -> list[Path]:
    files = [CSRC / s for s in SOURCES]
    files += sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))
    return files + [Path(__file__)]


def is_stale() -> bool:
    if not LIBRARY.exists():
        return True
    built = LIBRARY.stat().st_mtime
    return any(p.stat().st_mtime > built for p in _inputs())


def _compile(src: Path, obj: Path, verbose_ptxas: bool) -> None:
    cmd = [nvcc(), *GENCODE, *NVCC_FLAGS, "-c", str(src), "-o", str(obj)]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src.name}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)


def build(force: bool = False, verbose_ptxas: bool = False) -> Path:
    """Compile and link libgemm_tn.so if any source changed (or if forced)."""
    if not force and not verbose_ptxas and not is_stale():
        return LIBRARY
    BUILD_DIR.mkdir(parents=True, exist_ok=True)
    objs = [BUILD_DIR / (Path(s).stem + ".o") for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        list(pool.map(lambda so: _compile(CSRC / so[0], so[1], verbose_ptxas), zip(SOURCES, objs)))
    tmp = LIBRARY.with_name(f".libgemm_tn.{os.getpid()}.so")
    cmd = [nvcc(), *GENCODE, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-o", str(tmp)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ns = ap.parse_args()
    print(build(force=ns.force, verbose_ptxas=ns.ptxas_verbose))
