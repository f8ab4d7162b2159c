"""Builds ``libtopk_gb300.so`` in-tree from ``csrc/`` with nvcc for sm_103a."""

from __future__ import annotations

import os
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libtopk_gb300.so"

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC",
]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(home) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def build_library(out: Path = LIB, extra: list[str] | None = None, verbose: bool = False) -> Path:
    """Compile every .cu under csrc/ into one shared library."""
    tmp = out.with_name(out.name + f".{os.getpid()}.tmp")
    cmd = [nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", *(extra or []),
           *[str(s) for s in sources()], "-o", str(tmp)]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def needs_build(out: Path = LIB) -> bool:
    if not out.exists():
        return True
    t = out.stat().st_mtime
    deps = sources() + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    return any(d.stat().st_mtime > t for d in deps)


if __name__ == "__main__":
    build_library(verbose=True)
