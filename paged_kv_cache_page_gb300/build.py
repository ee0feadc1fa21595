"""Build libpagedattn.so (and the test-only libpa_selftest.so) in-tree with
nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into a shared
library with the CUDA runtime linked statically (no libcuda dependency at load
time; the driver is reached at first use).  Run ``python -m
paged_kv_cache_page_gb300.build`` or call :func:`build`.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libpagedattn.so"
SOURCES = ["api.cu", "append.cu", "decode.cu", "combine.cu", "noalloc.cu", "engine.cu",
           "rotary.cu", "prefill.cu"]
# Encoding self-test of the tensor-core operand layouts: test infrastructure,
# kept out of the product library.
SELFTEST_LIB = "libpa_selftest.so"
SELFTEST_SOURCES = ["selftest_tcgen05.cu", "selftest_tcgen05_t.cu",
                    "selftest_timeout.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path(name=LIB_NAME):
    return os.path.join(OUT_DIR, name)


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + list(extra)


def _compile(src, obj, extra, verbose):
    cmd = [nvcc_path(), "-c", os.path.join(CSRC, src), "-o", obj] + _flags(extra)
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _link(lib, objs):
    tmp = lib + ".tmp"
    cmd = [nvcc_path(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force=False, verbose=False, extra=()):
    """Compile (if needed) both libraries; return the path of libpagedattn.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "pagedattn.h"))
    targets = [(lib_path(LIB_NAME), SOURCES), (lib_path(SELFTEST_LIB), SELFTEST_SOURCES)]
    jobs, objs_of = [], {}
    for lib, sources in targets:
        objs_of[lib] = []
        for src in sources:
            obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
            objs_of[lib].append(obj)
            if force or verbose or _stale(obj, [os.path.join(CSRC, src)] + headers):
                jobs.append((src, obj))
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = [ex.submit(_compile, s, o, extra, verbose) for s, o in jobs]
            for f in futs:
                logs.append(f.result())
    for lib, objs in objs_of.items():
        if force or _stale(lib, objs):
            _link(lib, objs)
    if verbose:
        print("\n".join(logs))
    return lib_path(LIB_NAME)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
