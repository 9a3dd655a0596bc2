"""Build ``libsdv.so`` (the CUDA path, sm_103a) in-tree with nvcc.

Each translation unit compiles in parallel to an object under
``draft_verification_sdv_gb300/_build/``; the objects link into
``draft_verification_sdv_gb300/libsdv.so``.  Plain IEEE arithmetic (no
fast-math); ``-lineinfo`` for profiling.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsdv.so")
SOURCES = ["k1_rowpass.cu", "k2_select.cu", "k3_sample.cu", "k4_cps.cu", "k5_adl.cu", "sdv_api.cu", "sdv_static.cu"]
HEADERS = ["sdv_device.cuh", "sdv_plan.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    return ([os.path.join(CSRC, f) for f in SOURCES + HEADERS]
            + [os.path.join(ROOT, "include", "sdv.h"), os.path.abspath(__file__)])


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r.stdout + r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile libsdv.so if any source is newer than it; return its path."""
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in _deps()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        out = _run([nv] + flags + ["-c", os.path.join(CSRC, src), "-o", obj])
        return obj, out

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        for _, out in results:
            sys.stdout.write(out)
    tmp = LIB + ".tmp"
    _run([nv] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-lcudart"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
