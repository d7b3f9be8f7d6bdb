"""Build libqr.so in-tree with nvcc for sm_103a (no GPU needed to compile).

Each translation unit under csrc/ compiles in parallel; the objects link into
``libqr.so`` next to this file with the CUDA runtime linked statically and
every symbol hidden except the ``qr_*`` entry points of include/qr.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libqr.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["qr_capi.cu", "qr_grid.cu", "qr_encode.cu", "qr_decode.cu", "qr_reduce.cu", "qr_allreduce.cu",
           "qr_allreduce16_b3.cu", "qr_allreduce16_b4.cu", "qr_allreduce16_b6.cu", "qr_allreduce16_b8.cu",
           "qr_fc.cu", "qr_fc_allreduce_44.cu", "qr_fc_allreduce_48.cu", "qr_fc_allreduce_88.cu",
           "qr_twoshot.cu", "qr_twoshot_static.cu", "qr_twoshot_flags.cu", "qr_twoshot_peer.cu", "qr_timeouts.cu", "qr_fp4.cu",
           "qr_fc_twoshot.cu", "qr_fp4_twoshot.cu", "qr_codec_peer.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17",
    # every rounding step is an explicit _rn intrinsic; keep nvcc from fusing the rest
    "-fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqr.so")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "qr.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile csrc/*.cu into libqr.so (skipped when up to date).  Processes
    that build at the same time (the ranks of one job, parallel test
    workers) take turns on a lock file, and each re-checks whether the
    library is still stale once it holds the lock, so the objects are never
    written by two compilers at once."""
    if not force and not ptxas_info and not _stale():
        return LIB_PATH
    os.makedirs(OBJ_DIR, exist_ok=True)
    with open(os.path.join(OBJ_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and not ptxas_info and not _stale():
                return LIB_PATH
            return _build_locked(verbose, ptxas_info)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(verbose: bool, ptxas_info: bool) -> str:
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        return obj, p.stdout + p.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp] + [o for o, _ in results]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
