"""Build the library in-tree: csrc/*.cu and csrc/*.cpp -> _build/libfi.so (sm_103a only).

Translation units compile in parallel; the link is one nvcc call.  Runs the
same way on x86 (cross-compile, no GPU needed) and on the Arm GPU hosts.
Set FI_PTXAS_VERBOSE=1 to print register / shared-memory usage per kernel.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfi.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    srcs = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "fi.h"))
    return [os.path.join(CSRC, f) for f in srcs], headers


def _compile(src: str, obj: str, verbose: bool):
    nvcc = _nvcc()
    cmd = [nvcc, "-c", src, "-o", obj, "-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]
    if src.endswith(".cu"):
        cmd += ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]
        if verbose:
            cmd += ["-Xptxas", "-v"]
    else:
        cmd += ["-x", "c++"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr


def build(force: bool = False, verbose: bool | None = None) -> str:
    """Compile what changed and link; returns the library path.  Raises on any compiler error."""
    verbose = bool(int(os.environ.get("FI_PTXAS_VERBOSE", "0"))) if verbose is None else verbose
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "host_machine")
    machine = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != machine:
        force = True  # objects from another host architecture are never reused
        with open(stamp, "w") as f:
            f.write(machine + "\n")
    srcs, headers = _sources()
    newest_header = max(os.path.getmtime(h) for h in headers)
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s) + ".o")
        objs.append(o)
        if force or verbose or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), newest_header):
            jobs.append((s, o))
    errors = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, rc, out in ex.map(lambda j: _compile(j[0], j[1], verbose), jobs):
                if out.strip() and (rc != 0 or verbose):
                    sys.stderr.write(f"--- {os.path.basename(src)}\n{out}\n")
                if rc != 0:
                    errors.append(src)
    if errors:
        raise RuntimeError("compilation failed: " + ", ".join(os.path.basename(e) for e in errors))
    if jobs or not os.path.exists(LIB):
        cmd = [_nvcc(), "-shared", "-o", LIB] + objs + ARCH + ["-lcudart_static", "-ldl", "-lrt", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
