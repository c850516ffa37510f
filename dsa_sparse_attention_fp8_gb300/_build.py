"""In-tree build of libdsa_indexer.so (nvcc, sm_103a only)."""

from __future__ import annotations

import os
import platform
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB_DIR = PKG / "_lib"
LIB = LIB_DIR / "libdsa_indexer.so"
STAMP = LIB_DIR / "build.stamp"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa_indexer.so")


def _sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu")) + sorted(CSRC.glob("*.cuh")) + sorted(INCLUDE.glob("*.h"))


def _stamp_text() -> str:
    return f"{platform.machine()} {' '.join(ARCH_FLAGS)}"


def up_to_date() -> bool:
    if not LIB.exists() or not STAMP.exists():
        return False
    if STAMP.read_text().strip() != _stamp_text():
        return False
    t = LIB.stat().st_mtime
    return all(s.stat().st_mtime <= t for s in _sources())


def build_library(quiet: bool = False, force: bool = False) -> Path:
    """Compile csrc/dsa_indexer.cu into _lib/libdsa_indexer.so unless it is current."""
    if not force and up_to_date():
        return LIB
    LIB_DIR.mkdir(parents=True, exist_ok=True)
    tmp = LIB.with_suffix(f".so.tmp{os.getpid()}")
    cmd = [
        _nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17",
        "-Xcompiler", "-fPIC", "-shared", "-I", str(INCLUDE),
        "-o", str(tmp), str(CSRC / "dsa_indexer.cu"),
    ]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if not quiet and res.stderr.strip():
        print(res.stderr)
    os.replace(tmp, LIB)
    STAMP.write_text(_stamp_text())
    return LIB


if __name__ == "__main__":
    print(build_library(force=True))
