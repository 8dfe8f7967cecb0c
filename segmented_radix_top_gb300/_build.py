"""Builds libsegtopk.so from csrc/ with nvcc for sm_103a (in-tree, no cmake).

Each .cu is compiled to an object in parallel, then linked into one shared
library next to this file. A rebuild happens only when a source or header is
newer than the library.

The instrumented variant (libsegtopk_instr.so, variant="instr") is the same
sources compiled with SEGTOPK_STATS and SEGTOPK_TEST_HOOKS: per-CTA counters
(segtopk_read_stats) and the test hooks of the bounded copy wait
(segtopk_set_test_hooks). build_all() compiles both in one pool of
compiler processes.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libsegtopk.so")
VARIANTS = {
    "": (BUILD_DIR, LIB_PATH, []),
    "instr": (os.path.join(HERE, "_build_instr"), os.path.join(HERE, "libsegtopk_instr.so"),
              ["-DSEGTOPK_STATS", "-DSEGTOPK_TEST_HOOKS"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# hidden visibility: only the C ABI (SEGTOPK_API in include/segtopk.h) is
# exported, so two builds loaded in one process (the ordinary and the
# instrumented one) share no symbol, not even a function-local static
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE,
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def lib_path(variant: str = "") -> str:
    return VARIANTS[variant][1]


def up_to_date(variant: str = "") -> bool:
    path = lib_path(variant)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(variant: str, src: str, extra_flags, verbose: bool) -> str:
    build_dir, _, variant_flags = VARIANTS[variant]
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + variant_flags + list(extra_flags or []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def _link(variant: str, objs) -> str:
    out_path = VARIANTS[variant][1]
    tmp = out_path + ".tmp.%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + list(objs)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, out_path)
    return out_path


def build_variants(variants, force: bool = False, verbose: bool = False, extra_flags=None):
    """Builds the given variants, every translation unit of all of them in
    one pool of compiler processes; returns the library paths."""
    todo = [v for v in variants if force or not up_to_date(v)]
    for v in todo:
        os.makedirs(VARIANTS[v][0], exist_ok=True)
    srcs = _sources()
    jobs = [(v, s) for v in todo for s in srcs]
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            objs = list(ex.map(lambda j: _compile(j[0], j[1], extra_flags, verbose), jobs))
        for v in todo:
            _link(v, [o for (vv, _), o in zip(jobs, objs) if vv == v])
    return [lib_path(v) for v in variants]


def build(force: bool = False, verbose: bool = False, extra_flags=None, variant: str = "") -> str:
    return build_variants([variant], force=force, verbose=verbose, extra_flags=extra_flags)[0]


def build_all(force: bool = False, verbose: bool = False):
    """The library and its instrumented variant."""
    return build_variants(list(VARIANTS), force=force, verbose=verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else None,
                variant="instr" if "--instr" in sys.argv else ""))
