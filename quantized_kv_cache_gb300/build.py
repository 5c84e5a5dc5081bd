"""Build the in-tree shared library libkvq.so (CUDA for sm_103a) with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one link
step makes ``quantized_kv_cache_gb300/lib/libkvq.so``. The codec kernels are built with
``-fmad=false`` so that no multiply-add is contracted (their records must be reproducible
bit for bit); the host tables with ``-ffp-contract=off`` for the same reason.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
          "--expt-relaxed-constexpr"]
UNITS = {
    "kvq_api.cpp": [],
    "tables.cpp": [],
    "kernels_codec.cu": ["-fmad=false"],
    "kernels_seal.cu": ["-fmad=false"],
    "kernels_attn.cu": [],
    "kernels_body.cu": [],
    "synth.cu": [],
}


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


def _sources_newer_than(target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    for d in (CSRC, os.path.join(os.path.dirname(HERE), "include")):
        for f in os.listdir(d):
            if os.path.getmtime(os.path.join(d, f)) > t:
                return True
    return os.path.getmtime(__file__) > t


def build(force=False, verbose=False, ptxas_info=False):
    """Compile (if sources changed) and return the path of libkvq.so."""
    if not force and not _sources_newer_than(LIB):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def one(item):
        src, flags = item
        obj = os.path.join(BUILD_DIR, src + ".o")
        lang = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
        cmd = [cc] + lang + COMMON + ARCH + flags + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(one, UNITS.items()))
    objs = []
    for src, obj, r in results:
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        objs.append(obj)
    tmp = LIB + ".tmp"
    cmd = [cc, "-shared"] + ARCH + ["-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
