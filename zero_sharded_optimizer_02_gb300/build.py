"""Builds libzero.so in-tree: the CUDA kernels for sm_103a plus the host C++.

Two translation units are compiled in parallel and linked with the static
CUDA runtime, so the library loads without a GPU (symbol checks) and needs no
library path at run time.
"""
from __future__ import annotations

import os
import platform
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libzero.so")
BUILD = os.path.join(PKG, "_build", platform.machine())
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

SOURCES = {
    "zero_kernels.cu": ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
                        "-Xptxas", "-v", "-I", INCLUDE, "-c"],
    "zero_streamed.cu": ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler",
                         "-fPIC", "-Xptxas", "-v", "-I", INCLUDE, "-c"],
    "zero_gather.cu": ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
                       "-Xptxas", "-v", "-I", INCLUDE, "-c"],
    "zero_host.cpp": ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra", "-I", INCLUDE,
                      "-c"],
    "zero_checkpoint.cpp": ["g++", "-O2", "-std=c++17", "-fPIC", "-pthread", "-Wall",
                            "-Wextra", "-I", INCLUDE, "-c"],
}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def elf_matches_host(path: str) -> bool:
    """True if the ELF file at path was built for this machine's architecture."""
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return int.from_bytes(head[18:20], "little") == _ELF_MACHINE.get(platform.machine(), -1)


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target) or not elf_matches_host(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile what is stale and link libzero.so.  Extra nvcc flags (e.g. -D
    tuning macros of zero_kernels.cu) may be given in ZERO_NVCC_FLAGS, and an
    alternative source directory in ZERO_CSRC_DIR (for experiments kept out
    of the package); a change of either forces a rebuild."""
    os.makedirs(BUILD, exist_ok=True)
    extra = os.environ.get("ZERO_NVCC_FLAGS", "").split()
    csrc = os.environ.get("ZERO_CSRC_DIR") or CSRC
    stamp = os.path.join(BUILD, "nvcc_flags.txt")
    old = open(stamp).read() if os.path.exists(stamp) else None
    key = " ".join(extra) + ("" if csrc == CSRC else f" [csrc={csrc}]")
    if old != key:
        force = True
        with open(stamp, "w") as f:
            f.write(key)
    headers = [os.path.join(INCLUDE, "zero.h"), os.path.join(csrc, "zero_internal.h"),
               os.path.join(csrc, "zero_device.cuh"), os.path.join(csrc, "zero_ring.cuh"),
               os.path.join(csrc, "zero_small.cuh")]
    objs, procs = [], []
    for src, cmd in SOURCES.items():
        path = os.path.join(csrc, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *headers, __file__]):
            cmd = list(cmd)
            if cmd[0] == "nvcc":
                cmd = [_nvcc()] + cmd[1:] + extra
            log = open(obj + ".log", "w")
            procs.append((src, obj, log, subprocess.Popen(cmd + [path, "-o", obj], stdout=log,
                                                          stderr=subprocess.STDOUT)))
    failed = []
    for src, obj, log, p in procs:
        rc = p.wait()
        log.close()
        text = open(obj + ".log").read()
        if verbose or rc != 0:
            sys.stderr.write(f"--- {src} ---\n{text}")
        if rc != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"compilation failed: {failed}")
    if force or _stale(OUT, objs):
        tmp = OUT + f".tmp{os.getpid()}"
        subprocess.check_call([_nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-lpthread"])
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
