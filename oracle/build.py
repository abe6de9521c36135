"""Builds the CPU oracle (test infrastructure) into oracle/_build/libszoracle.so.

Plain gcc, one translation unit, no vector or threading flags.
"""
from __future__ import annotations

import os
import subprocess
from pathlib import Path

HERE = Path(__file__).resolve().parent
BUILD_DIR = HERE / "_build"
LIB_PATH = BUILD_DIR / "libszoracle.so"
SOURCES = [HERE / "sz_oracle.c"]
HEADERS = [HERE / "sz_oracle.h"]


def _stale(target: Path, deps: list[Path]) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, sources: list[Path] | None = None, out: Path | None = None) -> Path:
    """Compile the oracle shared library; returns its path.

    ``sources``/``out`` let a test compile a modified copy of the oracle into a
    scratch location without touching the real build.
    """
    srcs = list(sources) if sources is not None else SOURCES
    target = Path(out) if out is not None else LIB_PATH
    if not force and not _stale(target, srcs + HEADERS):
        return target
    target.parent.mkdir(parents=True, exist_ok=True)
    tmp = target.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", f"-I{HERE}", "-o", str(tmp)] + [str(s) for s in srcs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


if __name__ == "__main__":
    print(build(force=True))
