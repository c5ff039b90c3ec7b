"""Builds the CUDA library libg3h.so in-tree (bn254_scalar_field_gb300/_build/).

nvcc for sm_103a only; the C ABI is include/g3h.h. Run as
    python -m bn254_scalar_field_gb300.build
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libg3h.so")
SOURCES = [os.path.join(CSRC, "g3h.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("fr.cuh", "ntt.cuh", "kernels.cuh", "fq.cuh", "g1.cuh", "g2.cuh", "msm.cuh")] + [
    os.path.join(ROOT, "include", "g3h.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def source_digest():
    """SHA-256 (first 16 hex digits) of the CUDA sources and the ABI header: recorded next
    to profiler counters so that figures taken on older kernels are not reused."""
    import hashlib

    h = hashlib.sha256()
    for d in DEPS:
        with open(d, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_digest(kernel):
    """SHA-256 (first 16 hex digits) of the device code a profiled H-path kernel is built
    from (the NTT slice kernels: field arithmetic and ntt.cuh; the gather and join also
    kernels.cuh): recorded next to its profiler counters, so that figures taken on other
    code are not reused, while changes elsewhere keep them valid."""
    import hashlib

    files = ["fr.cuh", "ntt.cuh"]
    if not kernel.startswith("ntt_"):
        files.append("kernels.cuh")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def is_fresh():
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force=False, verbose=False):
    """Compile libg3h.so if it is missing or older than its sources; returns its path."""
    if not force and is_fresh():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v",
                             "-Xcompiler", "-fPIC", "-shared", "-o", tmp] + SOURCES
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(OUT_DIR, "ptxas.txt"), "w") as f:
        f.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stderr[-4000:])
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
