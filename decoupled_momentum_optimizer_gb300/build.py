"""Build libdemo_gb300.so in-tree for sm_103a (GB300) with nvcc.

Usage: ``python -m decoupled_momentum_optimizer_gb300.build`` (or ``build()``).
The translation units compile in parallel, then link into one shared
library next to this file.  The DCT factor header is regenerated from its
generator first, so the constants always come from gen_dct_factors.py.
"""

import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_NAME = "libdemo_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = ["demo_api.cu", "demo_step.cu", "demo_encode.cu", "demo_decode.cu", "demo_decode_lanes.cu",
           "demo_decode_groups.cu", "demo_dense.cu", "demo_adamw.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _regen_factors():
    gen = os.path.join(CSRC, "gen_dct_factors.py")
    out = subprocess.run([sys.executable, gen], check=True, capture_output=True, text=True).stdout
    path = os.path.join(CSRC, "dct32_factors.cuh")
    old = open(path).read() if os.path.exists(path) else None
    if old != out:
        with open(path, "w") as f:
            f.write(out)


def _compile(src, build_dir, verbose):
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False, force=False):
    """Compile and link the library; returns its path."""
    _regen_factors()
    build_dir = os.path.join(os.path.dirname(HERE), "_build")
    os.makedirs(build_dir, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "demo.h")]
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(d) for d in deps)
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, build_dir, verbose), SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB_PATH + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
