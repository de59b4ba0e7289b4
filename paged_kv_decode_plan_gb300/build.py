"""Builds ``libpkd.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: ``python -m paged_kv_decode_plan_gb300.build [--force] [--verbose]``.
Translation units compile in parallel into ``_build/``; the shared library is
written next to this file.
"""
from __future__ import annotations

import argparse
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build", platform.machine())
LIB_PATH = os.path.join(HERE, "libpkd.so")

SOURCES = ["plan.cpp", "api.cu", "decode.cu", "merge.cu", "prefix.cu", "append.cu",
           "static_scratch.cu", "plan_copy.cu"]
HEADERS = ["pkd_internal.h", "ptx.cuh", "kernel_common.cuh", "tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _native(path: str) -> bool:
    """True when the ELF file's machine field matches this host."""
    machines = {"x86_64": 62, "aarch64": 183}
    want = machines.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if want is None or len(head) < 20:
        return True
    return int.from_bytes(head[18:20], "little") == want


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(INCLUDE, "pkd.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + headers):
            flags = list(COMMON) + list(extra)
            if src.endswith(".cu"):
                flags += ARCH
                if verbose:
                    flags += ["-Xptxas", "-v"]
            jobs.append([nvcc()] + flags + ["-c", path, "-o", obj])

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("compile failed:\n%s\n%s\n%s" %
                               (" ".join(cmd), res.stdout, res.stderr))
        return res.stderr

    if jobs:
        with ThreadPoolExecutor(len(jobs)) as pool:
            logs = list(pool.map(run, jobs))
        if verbose:
            for log in logs:
                print(log)
    if force or jobs or _stale(LIB_PATH, objs) or not _native(LIB_PATH):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static"]
        run(cmd)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
