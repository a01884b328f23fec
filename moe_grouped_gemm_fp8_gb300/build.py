"""Builds ``libdg.so`` (the CUDA library behind include/dg.h) in-tree.

Each translation unit is compiled by nvcc for sm_103a in parallel, then
linked into one shared library next to this file.  No CMake, no torch
extension machinery: the library has a plain C ABI.

``build(debug=True)`` builds ``libdg_debug.so`` beside it from the same
sources with ``-DDG_DEBUG_CHECKS=1``: the kernels check their load
coordinates, TMEM columns, store rows and stream-K slots, and record
DG_ERR_DEVICE_CHECK with the site in the error word instead of trapping.
The binding loads it when ``DG_DEBUG_LIBRARY=1``.

``build_floor()`` builds ``libdg_floor.so``, a measurement aid for the
benchmark (the per-launch time of a plain streaming read from HBM), apart
from the GEMM library.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdg.so")
DEBUG_LIB = os.path.join(HERE, "libdg_debug.so")
FLOOR_LIB = os.path.join(HERE, "libdg_floor.so")
FLOOR_SRC = os.path.join(CSRC, "hbm_floor.cu")

SOURCES = ["gemm_bn128.cu", "gemm_bn192.cu", "gemm_bn224.cu", "gemm_bn256.cu",
           "gemm2_bn192.cu", "gemm2_bn224.cu", "gemm2_bn256.cu", "gemm_splitk.cu", "gemm_tall.cu", "gemm_promote.cu", "gemm_decode.cu", "gemm_kgrouped.cu", "gemm.cu",
           "quant.cu", "host.cu", "static_ws.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "dg.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, lineinfo: bool = True, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and not _stale(lib):
        return lib
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"]
    if debug:
        flags.append("-DDG_DEBUG_CHECKS=1")
    if lineinfo:
        flags.append("-lineinfo")
    if verbose:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src + ".o")
        objs.append(obj)
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((cmd, text))
        elif verbose and text:
            sys.stderr.write(text)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + t for c, t in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = lib + ".tmp%d" % os.getpid()
    subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, lib)
    return lib


def build_floor(force: bool = False) -> str:
    """libdg_floor.so: the streaming-read floor kernel the benchmark times."""
    if not force and os.path.exists(FLOOR_LIB) and os.path.getmtime(FLOOR_LIB) >= max(
            os.path.getmtime(FLOOR_SRC), os.path.getmtime(os.path.abspath(__file__))):
        return FLOOR_LIB
    tmp = FLOOR_LIB + ".tmp%d" % os.getpid()
    subprocess.run([_nvcc()] + ARCH + ["-O3", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, FLOOR_SRC], check=True)
    os.replace(tmp, FLOOR_LIB)
    return FLOOR_LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
