"""Build libzero (the CUDA library behind include/zero.h) in-tree for sm_103a.

    python -m zero_partitioned_mixed_flat_gb300.build [--force]

Compiles csrc/*.cu and csrc/*.cpp with nvcc in parallel and links
zero_partitioned_mixed_flat_gb300/_lib/libzero.so (CUDA runtime linked
statically, so the library loads without a GPU; device calls need one).
"""
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libzero.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libzero")


COMMON = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC,-ffp-contract=off,-Wall",
          "-I", INCLUDE, "-I", CSRC]
DEVICE = ARCH + ["-lineinfo", "--fmad=false", "-Xptxas", "-warn-spills"]


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _fingerprint(srcs) -> str:
    h = hashlib.sha256()
    for f in srcs + sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".h")) \
            + [os.path.join(INCLUDE, "zero.h"), os.path.abspath(__file__)]:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(COMMON + DEVICE).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = _sources()
    fp = _fingerprint(srcs)
    stamp = os.path.join(OUT_DIR, "libzero.stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tool = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
        cmd = [tool, *COMMON, "-c", src, "-o", obj]
        if src.endswith(".cu"):
            cmd[1:1] = DEVICE
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [tool, "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
