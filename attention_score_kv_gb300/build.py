"""Build libkvc.so in-tree from csrc/ for GB300 (sm_103a).

Each translation unit is compiled by nvcc in parallel, then linked into
``attention_score_kv_gb300/libkvc.so`` (static CUDA runtime).  Run
``python -m attention_score_kv_gb300.build`` or call :func:`build`.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvc.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, " ".join(cmd), p.stdout


def build(verbose: bool = False, extra_flags=None, force: bool = False, lib_path: str | None = None,
          build_dir: str | None = None) -> str:
    """Compile csrc/*.cu for sm_103a and link libkvc.so; returns its path.

    ``extra_flags`` are appended to every nvcc compile; ``lib_path`` and
    ``build_dir`` place the library and objects elsewhere (default: in-tree).
    """
    nvcc = _nvcc()
    LIB = lib_path or globals()["LIB"]
    BUILD = build_dir or globals()["BUILD"]
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(HERE, "..", "include", "kvc.h"))
    newest_hdr = max(os.path.getmtime(h) for h in headers)
    extra = list(extra_flags or [])
    jobs, objs = [], []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), newest_hdr):
            jobs.append([nvcc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for rc, cmd, out in ex.map(_run, jobs):
            if verbose or rc:
                sys.stderr.write(f"{cmd}\n{out}")
            if rc:
                raise RuntimeError(f"nvcc failed:\n{cmd}\n{out}")
    if jobs or not os.path.exists(LIB):
        tmp = LIB + ".tmp"
        rc, cmd, out = _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        if verbose or rc:
            sys.stderr.write(f"{cmd}\n{out}")
        if rc:
            raise RuntimeError(f"link failed:\n{cmd}\n{out}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="--force" in sys.argv))
