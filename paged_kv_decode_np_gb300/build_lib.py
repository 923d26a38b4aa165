"""Build libnp_paged.so for sm_103a with nvcc (in-tree, no cmake).

The decode kernel is compiled once per (storage dtype, head_dim) from
``csrc/decode_inst.cu`` with -D flags; every object compiles in parallel and
links into one shared library with the CUDA runtime linked statically.
``python -m paged_kv_decode_np_gb300.build_lib [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libnp_paged.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
HEAD_DIMS = (16, 32, 64, 128, 256)


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return cand


def _units(extra: list[str], build_dir: str, csrc: str) -> list[tuple[str, str, list[str]]]:
    """(source, object, extra flags) for every translation unit."""
    objdir = os.path.join(build_dir, "obj")
    units = [
        (os.path.join(csrc, "api.cu"), os.path.join(objdir, "api.o"), []),
        (os.path.join(csrc, "append_reduce.cu"), os.path.join(objdir, "append_reduce.o"), []),
        (os.path.join(csrc, "noalloc.cu"), os.path.join(objdir, "noalloc.o"), []),
    ]
    for bf16 in (0, 1):
        for d in HEAD_DIMS:
            name = f"decode_{'bf16' if bf16 else 'f32'}_d{d}.o"
            units.append((os.path.join(csrc, "decode_inst.cu"), os.path.join(objdir, name),
                          [f"-DNPK_BF16={bf16}", f"-DNPK_D={d}"]))
    return [(s, o, ["-I", csrc] + f + extra) for s, o, f in units]


def _deps(csrc: str) -> list[str]:
    files = [os.path.join(csrc, f) for f in os.listdir(csrc)]
    files.append(os.path.join(INCLUDE, "np_paged.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, flags: list[str], verbose_ptxas: bool) -> str:
    cmd = [nvcc(), "-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, *flags, "-c", src, "-o", obj + ".tmp"]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{p.stderr}")
    os.replace(obj + ".tmp", obj)
    return p.stderr


def build(force: bool = False, extra_flags: list[str] | None = None, out: str | None = None,
          verbose_ptxas: bool = False, jobs: int | None = None,
          build_dir: str | None = None, csrc: str | None = None) -> str:
    """Compile (incrementally) and link; returns the library path.

    ``extra_flags`` (e.g. -D tuning macros) or another source directory
    ``csrc`` need their own ``build_dir`` and ``out`` so they never mix with
    the default build's objects.
    """
    out = out or LIB
    build_dir = build_dir or BUILD
    csrc = csrc or CSRC
    extra = list(extra_flags or [])
    if (extra or csrc != CSRC) and build_dir == BUILD:
        raise ValueError("extra_flags / csrc need a separate build_dir")
    units = _units(extra, build_dir, csrc)
    os.makedirs(os.path.join(build_dir, "obj"), exist_ok=True)
    deps = _deps(csrc)
    todo = [u for u in units if force or _stale(u[1], deps)]
    logs = {}
    if todo:
        jobs = jobs or min(len(todo), max(1, os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(jobs) as ex:
            futs = {ex.submit(_compile, s, o, f, verbose_ptxas): o for s, o, f in todo}
            for fut in cf.as_completed(futs):
                logs[futs[fut]] = fut.result()
    objs = [o for _, o, _ in units]
    if todo or _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stderr}")
        os.replace(tmp, out)
    if verbose_ptxas:
        for o in sorted(logs):
            print(f"== {os.path.basename(o)}\n{logs[o]}")
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
