"""Builds ``libtopk_gb300.so`` in-tree from ``csrc/`` with nvcc for sm_103a.

Two instrumented variants come from the same sources with one macro each:
``libtopk_gb300_timeline.so`` (``-DTOPK_TIMELINE=1``: per-CTA global-timer
stamps, read with ``topk_timeline_read``; level 2 adds per-activity cycle
counts, which slow the filter loop) and
``libtopk_gb300_debug.so`` (``-DTOPK_DEBUG_BOUNDS=1``: every shared- and
global-memory index the selection computes is checked before use; a bad one
sets ``TOPK_STATUS_BOUNDS`` and the access is skipped).  The product library
is the plain one.
"""

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

VARIANTS = {
    "timeline": ["-DTOPK_TIMELINE=1"],
    "debug": ["-DTOPK_DEBUG_BOUNDS=1"],
}


def variant_path(name: str) -> Path:
    return PKG / f"libtopk_gb300_{name}.so"


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(home) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _command(out: Path, extra: list[str] | None) -> tuple[list[str], Path]:
    tmp = out.with_name(out.name + f".{os.getpid()}.tmp")
    cmd = [nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", *(extra or []),
           *[str(s) for s in sources()], "-o", str(tmp)]
    return cmd, tmp


def build_library(out: Path = LIB, extra: list[str] | None = None, verbose: bool = False) -> Path:
    """Compile every .cu under csrc/ into one shared library."""
    cmd, tmp = _command(out, extra)
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_variant(name: str, verbose: bool = False) -> Path:
    return build_library(variant_path(name), VARIANTS[name], verbose)


def build_all(verbose: bool = False) -> list[Path]:
    """The product library and both instrumented variants, compiled in
    parallel (one nvcc each)."""
    jobs = [(LIB, None)] + [(variant_path(v), f) for v, f in VARIANTS.items()]
    procs = []
    for out, extra in jobs:
        cmd, tmp = _command(out, extra)
        if verbose:
            print(" ".join(cmd))
        procs.append((subprocess.Popen(cmd), tmp, out))
    failed = []
    for proc, tmp, out in procs:
        if proc.wait() != 0:
            failed.append(out.name)
        else:
            os.replace(tmp, out)
    if failed:
        raise RuntimeError(f"nvcc failed for {', '.join(failed)}")
    return [out for _, _, out in procs]


def needs_build(out: Path = LIB) -> bool:
    if not out.exists():
        return True
    t = out.stat().st_mtime
    deps = sources() + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    return any(d.stat().st_mtime > t for d in deps)


if __name__ == "__main__":
    build_all(verbose=True)
