"""CPU oracle for segmented top-k (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library: it has
its own type codes, its own build step and its own ctypes binding.

The arithmetic lives in ``oracle.c`` (plain C, numeric key comparison, merge
sort); this module only builds it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

# Type codes of this oracle (independent of the CUDA library's enums).
DTYPES = {"f16": 0, "bf16": 1, "f32": 2, "f64": 3, "u32": 4, "i32": 5}
NUMPY_STORAGE = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32,
                 "f64": np.uint64, "u32": np.uint32, "i32": np.int32}
DIRECTIONS = {"max": 0, "min": 1}
TIE_BREAKS = {"unspecified": 0, "prefer_smaller_index": 1, "prefer_larger_index": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no GPU needed)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load(path: str):
    L = ctypes.CDLL(path)
    L.oracle_batched_topk.restype = ctypes.c_int
    L.oracle_batched_topk.argtypes = [
        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    L.oracle_decode_f16.restype = ctypes.c_double
    L.oracle_decode_f16.argtypes = [ctypes.c_uint32]
    L.oracle_decode_bf16.restype = ctypes.c_double
    L.oracle_decode_bf16.argtypes = [ctypes.c_uint32]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(build())
    return _lib


def use_library(path: str | None):
    """Point this binding at another build of the oracle (the mutation test
    compiles deliberately broken copies of oracle.c); None restores the
    default library."""
    global _lib
    _lib = None if path is None else _load(path)


def _ptr(a):
    return None if a is None else a.ctypes.data


def batched_topk(dtype: str, keys: np.ndarray, values, offsets: np.ndarray, k: int,
                 direction: str, tie_break: str, out_keys: np.ndarray | None = None,
                 out_values: np.ndarray | None = None, threads: int = 1,
                 seg_range: tuple[int, int] | None = None):
    """Run the oracle; returns (out_keys, out_values) laid out [num_segments, k].

    ``keys`` holds raw bit patterns (the storage dtype of NUMPY_STORAGE).
    Slots past min(k, n) keep whatever ``out_keys``/``out_values`` held.
    ``threads`` > 1 splits the segments over a thread pool (the C call
    releases the GIL), which changes nothing in the result.
    """
    L = lib()
    keys = np.ascontiguousarray(keys, dtype=NUMPY_STORAGE[dtype])
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    num_segments = offsets.shape[0] - 1
    if values is not None:
        values = np.ascontiguousarray(values, dtype=np.int32)
    if out_keys is None:
        out_keys = np.zeros(num_segments * k, dtype=NUMPY_STORAGE[dtype])
    if out_values is None and values is not None:
        out_values = np.zeros(num_segments * k, dtype=np.int32)
    lo, hi = seg_range if seg_range is not None else (0, num_segments)

    def run(a, b):
        rc = L.oracle_batched_topk(DTYPES[dtype], _ptr(keys), _ptr(values), _ptr(offsets),
                                   a, b, k, DIRECTIONS[direction], TIE_BREAKS[tie_break],
                                   _ptr(out_keys), _ptr(out_values))
        if rc != 0:
            raise RuntimeError("oracle failed with code %d" % rc)

    if threads <= 1 or hi - lo < 2:
        run(lo, hi)
    else:
        # balance by key count: cut the segment range at equal prefix sums
        lens = np.maximum(offsets[lo + 1:hi + 1] - offsets[lo:hi], 0)
        csum = np.concatenate([[0], np.cumsum(lens)])
        parts = max(1, min(threads * 4, hi - lo))
        cuts = np.searchsorted(csum, np.linspace(0, csum[-1], parts + 1)).tolist()
        cuts[0], cuts[-1] = 0, hi - lo
        bounds = sorted(set(cuts))
        with ThreadPoolExecutor(max_workers=threads) as ex:
            futs = [ex.submit(run, lo + a, lo + b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
            for f in futs:
                f.result()
    return out_keys, out_values


def decode_f16(bits: int) -> float:
    return lib().oracle_decode_f16(bits)


def decode_bf16(bits: int) -> float:
    return lib().oracle_decode_bf16(bits)
