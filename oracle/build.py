"""Build step for the CPU oracle's C part (test infrastructure).

Compiles ``gemm_oracle.c`` and ``attention_oracle.c`` into
``oracle/liboracle_<machine>.so`` with gcc: -O2, no fast-math and
-ffp-contract=off, so the fp64 loops round exactly as their source reads on
both x86_64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import platform
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
SOURCES = (HERE / "gemm_oracle.c", HERE / "attention_oracle.c")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def library_path(plant: int = 0, out_dir: Path | None = None) -> Path:
    tag = platform.machine()
    name = f"liboracle_{tag}.so" if plant == 0 else f"liboracle_{tag}_plant{plant}.so"
    return (out_dir or HERE) / name


def build(plant: int = 0, out_dir: Path | None = None, force: bool = False) -> Path:
    """Compile the oracle library (``plant`` > 0 builds a deliberately wrong
    variant for the pinning tests). Returns the path of the shared object."""
    out = library_path(plant, out_dir)
    if (not force and out.exists()
            and all(out.stat().st_mtime >= src.stat().st_mtime for src in SOURCES)):
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".tmp{os.getpid()}.so")
    cmd = ["gcc", *CFLAGS, f"-DORACLE_PLANT={int(plant)}", *map(str, SOURCES), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
