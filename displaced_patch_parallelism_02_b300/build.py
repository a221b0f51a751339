"""Builds libdpp.so in-tree with nvcc for sm_103a (B300).

    python displaced_patch_parallelism_02_b300/build.py [--force] [--verbose-ptxas]

(run it by path: importing the package first would load the library that is
about to be rebuilt)

Each translation unit in csrc/ is compiled to an object under
csrc/_build/ in parallel, then linked into libdpp.so next to this file.
A SHA-256 of the sources, headers and compiler flags is compiled into the
library (dpp_source_hash()); a library whose hash differs from the current
sources is rebuilt whatever its file times say, and objects are reused only
when newer than their sources and built with the same hash.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(CSRC, "_build")
LIB = os.path.join(PKG, "libdpp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "dpp.h")]


def source_hash() -> str:
    """SHA-256 of every source, header and the compiler flags."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(CSRC, "*.cu"))) + sorted(_headers()):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


def library_hash(lib: str = LIB):
    """The hash compiled into an existing libdpp.so, read in a child process
    (so this process does not keep the library loaded), or None."""
    if not os.path.exists(lib):
        return None
    code = ("import ctypes, sys; l = ctypes.CDLL(sys.argv[1]); "
            "f = l.dpp_source_hash; f.restype = ctypes.c_char_p; print(f().decode())")
    r = subprocess.run([sys.executable, "-c", code, lib], capture_output=True, text=True)
    return r.stdout.strip() if r.returncode == 0 else None


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    want = source_hash()
    stamp = os.path.join(BUILD, "source_hash")
    built_with = open(stamp).read().strip() if os.path.exists(stamp) else None
    if built_with != want:  # objects from other sources or flags: rebuild them all
        force = True
    if not force and library_hash() != want:
        force = True  # a library whose embedded hash does not match these sources
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc()] + ARCH + FLAGS + [f"-DDPP_SOURCE_SHA256=\"{want}\""] + \
                (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", s, "-o", o]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        for cmd, r in ex.map(run, jobs):
            out = (r.stdout + r.stderr).strip()
            if r.returncode != 0:
                failed.append((cmd, out))
            elif out and (verbose_ptxas or not quiet):
                print(out)
    if failed:
        for cmd, out in failed:
            sys.stderr.write(" ".join(cmd) + "\n" + out + "\n")
        raise RuntimeError(f"nvcc failed for {len(failed)} translation unit(s)")
    if force or jobs or _stale(LIB, objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", LIB] + objs + ["-lcudart_static", "-lrt",
                                                                 "-ldl", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    with open(stamp, "w") as fh:
        fh.write(want)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas, quiet=False))


if __name__ == "__main__":
    main()
