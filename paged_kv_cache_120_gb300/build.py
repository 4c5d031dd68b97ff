"""Build libpa.so in-tree for sm_103a (nvcc for the CUDA unit, g++ for host C++).

Usage: ``python -m paged_kv_cache_120_gb300.build [--force] [--verbose]``.
Translation units compile in parallel; the result is
``paged_kv_cache_120_gb300/_build/libpa.so``.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpa.so")
HEADER = os.path.join(ROOT, "include", "pa.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"] + ARCH
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-Wall", "-Wextra"]

UNITS = [
    ("pa_kernels.cu", "nvcc"),
    ("pa_prefill.cu", "nvcc"),
    ("pa_static_scratch.cu", "nvcc"),
    ("block_allocator.cpp", "g++"),
    ("prefix_cache.cpp", "g++"),
    ("pa_errors.cpp", "g++"),
]


def _sources():
    files = [os.path.join(CSRC, f) for f, _ in UNITS]
    files += [os.path.join(CSRC, "pa_internal.h"), os.path.join(CSRC, "pa_device.cuh"), HEADER,
              os.path.abspath(__file__)]
    return files


def _fingerprint(extra: list[str]) -> str:
    h = hashlib.sha256()
    for f in _sources():
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(extra).encode())
    return h.hexdigest()


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, extra_nvcc: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Compile and link libpa.so into ``out_dir`` (default: the in-tree _build)."""
    extra_nvcc = list(extra_nvcc or [])
    build_dir = out_dir or BUILD
    lib_path = os.path.join(build_dir, "libpa.so")
    os.makedirs(build_dir, exist_ok=True)
    stamp = os.path.join(build_dir, "libpa.stamp")
    fp = _fingerprint(extra_nvcc)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return lib_path
    nvcc = _nvcc()

    def compile_unit(unit):
        name, tool = unit
        src = os.path.join(CSRC, name)
        obj = os.path.join(build_dir, name + ".o")
        if tool == "nvcc":
            cmd = [nvcc] + NVCC_FLAGS + extra_nvcc + ["-c", src, "-o", obj]
            if verbose:
                cmd += ["-Xptxas", "-v"]
        else:
            cmd = ["g++"] + CXX_FLAGS + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(fp)
    return lib_path


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    main()
