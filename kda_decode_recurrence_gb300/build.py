"""Build libkda.so in-tree with nvcc for sm_103a (GB300).

The translation units are compiled in parallel and linked into
``kda_decode_recurrence_gb300/_build/libkda.so`` against the shared CUDA
runtime (the same libcudart PyTorch loads).  Two variant libraries are
linked from the same objects with one translation unit recompiled:

  libkda_outgate_swish.so  the fused block's output gate compiled as swish
                           (z * sigmoid(z)) instead of sigmoid
  libkda_testhooks.so      test-only: the decode kernel's copy-wait limit and
                           one withheld work item are settable
                           (kda_test_set_decode_hooks), to exercise its
                           timeout report without a fault

Usage:

    python -m kda_decode_recurrence_gb300.build [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libkda.so")
# Library variants: name -> (library path, {source recompiled: extra nvcc flags})
VARIANTS = {
    "outgate_swish": (os.path.join(BUILD_DIR, "libkda_outgate_swish.so"),
                      {"kda_block.cu": ["-DKDA_BLOCK_OUTPUT_GATE_SWISH=1"]}),
    "debugbounds": (os.path.join(BUILD_DIR, "libkda_debugbounds.so"),
                    {f: ["-DKDA_DEBUG_BOUNDS=1"] for f in ("kda_decode.cu", "kda_prefill.cu",
                                                          "kda_block.cu")}),
    "testhooks": (os.path.join(BUILD_DIR, "libkda_testhooks.so"),
                  {"kda_decode.cu": ["-DKDA_TEST_HOOKS=1"], "kda_prefill.cu": ["-DKDA_TEST_HOOKS=1"]}),
}

SOURCES = ["kda_api.cu", "kda_decode.cu", "kda_block.cu", "kda_tc_gemm.cu", "kda_block_static.cu", "kda_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda")
    return cand


def _cuda_lib_dir() -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(_nvcc())))
    for sub in ("lib64", "lib"):
        d = os.path.join(root, sub)
        if os.path.isdir(d):
            return d
    return "/usr/local/cuda/lib64"


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files


def _up_to_date() -> bool:
    libs = [LIB_PATH] + [v[0] for v in VARIANTS.values()]
    if not all(os.path.exists(p) for p in libs):
        return False
    t = min(os.path.getmtime(p) for p in libs)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libkda.so and its variants; returns libkda.so's path.
    Raises on failure."""
    if not force and _up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(job):
        src, tag, extra = job
        obj = os.path.join(BUILD_DIR, src.replace(".cu", f"{tag}.o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}{tag}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    jobs = [(src, "", []) for src in SOURCES]
    jobs += [(src, f"_{name}", flags) for name, (_, per_src) in VARIANTS.items()
             for src, flags in per_src.items()]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    base = objs[:len(SOURCES)]

    def link(objects, path):
        tmp = path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objects, "-o", tmp,
               "-Xlinker", f"-rpath={_cuda_lib_dir()}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)

    link(base, LIB_PATH)
    for name, (path, per_src) in VARIANTS.items():
        swap = {os.path.join(BUILD_DIR, src.replace(".cu", ".o")):
                os.path.join(BUILD_DIR, src.replace(".cu", f"_{name}.o")) for src in per_src}
        link([swap.get(o, o) for o in base], path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
