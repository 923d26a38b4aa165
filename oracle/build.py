"""Compile the C oracle into a shared library (test infrastructure).

Run as ``python -m oracle.build``; ``__graft_entry__.build()`` and the test
suite call :func:`build` too.  Plain gcc, no vendor code, the same flags on
x86-64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import sys
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libnp_oracle.so")
SOURCES = [os.path.join(HERE, "np_oracle.c")]
DEPS = SOURCES + [os.path.join(HERE, "decode_body.h")]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def compile_oracle(sources: list[str], out_path: str) -> None:
    """gcc -O2 (no fast-math: libm exp/log and IEEE arithmetic as written)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}.{threading.get_ident()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, *sources, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)


_LOCK = threading.Lock()


def build(force: bool = False) -> str:
    with _LOCK:  # threads of one process build it once
        if force or _stale(LIB_PATH, DEPS):
            compile_oracle(SOURCES, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
