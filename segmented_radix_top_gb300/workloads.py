"""Seeded synthetic workloads for segmented top-k.

This module only draws inputs. It contains none of the selection arithmetic,
and both the CUDA path and the CPU oracle read the arrays it returns.

Keys are returned as raw bit patterns in their storage type (uint16 for
f16/bf16, uint32 for f32/u32, int32 for i32, uint64 for f64), so that +0.0 and
-0.0 stay distinguishable everywhere.

The five named workloads follow the shapes the pages benchmark (fixed and
variable segment sizes, keys and pairs, tie-heavy inputs; "Implement Segmented
TopK using Thread-Block-Clusters", section 9 "Testing", and "Fix BlockTopK
+/-0.0 handling", test helpers with +/-0.0 and +/-inf boundary keys). There is
no public dataset; every array is drawn from numpy's PCG64 with seed
1000 + workload number, so both sides see identical bytes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

STORAGE = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32,
           "f64": np.uint64, "u32": np.uint32, "i32": np.int32}
KEY_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "f64": 8, "u32": 4, "i32": 4}


@dataclass
class Workload:
    name: str
    dtype: str                 # key type name
    keys: np.ndarray           # raw key bits, storage dtype
    values: np.ndarray | None  # int32 payload or None (keys only)
    offsets: np.ndarray        # int64, num_segments + 1
    k: int
    direction: str             # "max" | "min"
    determinism: str           # "not_guaranteed" | "run_to_run" | "gpu_to_gpu"
    tie_break: str             # "unspecified" | "prefer_smaller_index" | "prefer_larger_index"
    ordering: str              # "unsorted" | "sorted" | "stable_sorted"
    info: dict = field(default_factory=dict)

    @property
    def num_segments(self) -> int:
        return int(self.offsets.shape[0] - 1)

    @property
    def num_keys(self) -> int:
        return int(self.keys.shape[0])

    @property
    def lengths(self) -> np.ndarray:
        return np.maximum(np.diff(self.offsets), 0)

    @property
    def max_segment_len(self) -> int:
        return int(self.lengths.max()) if self.num_segments else 0


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def f64_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)


def f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float16).view(np.uint16)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit patterns (NaN kept NaN)."""
    w = f32_bits(x).astype(np.uint64)
    lsb = (w >> 16) & 1
    r = ((w + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r[nan] = ((w[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def offsets_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)


# --------------------------------------------------------------------------
# The five benchmark workloads. `segments` / `seg_len` shrink a workload for
# parity tests while keeping its structure (value distribution, ties, mode).
# --------------------------------------------------------------------------

def workload1(segments: int = 16, max_len: int = 4096) -> Workload:
    """16 segments, lengths uniform in [1, 4096]; fp32 uniform in [-1, 1] with
    10% of entries replaced by +0.0 or -0.0 (sign 50/50); k=8, max, keys only,
    gpu_to_gpu + prefer_smaller_index + stable_sorted."""
    g = _rng(1001)
    lengths = g.integers(1, max_len + 1, size=segments)
    n = int(lengths.sum())
    x = g.uniform(-1.0, 1.0, size=n).astype(np.float32)
    z = g.random(n) < 0.10
    neg = g.random(n) < 0.5
    x[z & neg] = np.float32(-0.0)
    x[z & ~neg] = np.float32(0.0)
    return Workload("fp32 ragged <=4096, k=8 max keys (+/-0 ties)", "f32", f32_bits(x), None,
                    offsets_from_lengths(lengths), 8, "max", "gpu_to_gpu",
                    "prefer_smaller_index", "stable_sorted")


def workload2(segments: int = 128, seg_len: int = 152064) -> Workload:
    """128 x 152064 fp32 ~ N(0,1) (logit rows); k=50, max, pairs with value =
    local source index, gpu_to_gpu + prefer_smaller_index + stable_sorted."""
    g = _rng(1002)
    x = g.standard_normal(size=segments * seg_len, dtype=np.float32)
    vals = np.tile(np.arange(seg_len, dtype=np.int32), segments)
    return Workload("fp32 %d x %d N(0,1), k=50 max pairs" % (segments, seg_len), "f32",
                    f32_bits(x), vals, offsets_from_lengths([seg_len] * segments), 50, "max",
                    "gpu_to_gpu", "prefer_smaller_index", "stable_sorted")


def workload3(segments: int = 10000, max_len: int = 65536) -> Workload:
    """10000 segments with log-uniform lengths in [1, 65536]; fp16 keys on 256
    levels (j - 128)/32, j uniform in [0, 256), with j = 128 written as +0.0 or
    -0.0 (50/50), so heavy ties; k=32, min, pairs (random int32),
    gpu_to_gpu + prefer_larger_index, unsorted."""
    g = _rng(1003)
    lengths = np.floor(np.exp(g.uniform(0.0, np.log(max_len + 1), size=segments)))
    lengths = np.clip(lengths, 1, max_len).astype(np.int64)
    n = int(lengths.sum())
    j = g.integers(0, 256, size=n)
    x = ((j - 128) / 32.0).astype(np.float16)
    bits = f16_bits(x).copy()
    zero = j == 128
    negz = g.random(n) < 0.5
    bits[zero & negz] = 0x8000
    bits[zero & ~negz] = 0x0000
    vals = g.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
    return Workload("fp16 %d log-uniform <=%d, 256 levels, k=32 min pairs" % (segments, max_len),
                    "f16", bits, vals, offsets_from_lengths(lengths), 32, "min", "gpu_to_gpu",
                    "prefer_larger_index", "unsorted")


BOUNDARY_U32 = 0xFFC00000


def workload4(segments: int = 64, seg_len: int = 1048576) -> Workload:
    """64 x 1,048,576 uint32; half of each segment's positions (a seeded
    shuffle) hold one boundary value 0xFFC00000 and the rest are uniform over
    [0, 2^32). About 512 uniform keys per segment lie above the boundary, so the
    1024th key falls inside the tie block. k=1024, max, pairs (random int32),
    gpu_to_gpu + prefer_smaller_index + stable_sorted."""
    g = _rng(1004)
    keys = g.integers(0, 2**32, size=(segments, seg_len), dtype=np.uint64).astype(np.uint32)
    half = seg_len // 2
    for s in range(segments):
        pos = g.permutation(seg_len)[:half]
        keys[s, pos] = BOUNDARY_U32
    vals = g.integers(-2**31, 2**31, size=segments * seg_len, dtype=np.int64).astype(np.int32)
    return Workload("u32 %d x %d half ties, k=1024 max pairs" % (segments, seg_len), "u32",
                    keys.reshape(-1), vals, offsets_from_lengths([seg_len] * segments), 1024,
                    "max", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted")


def workload5(segments: int = 4096, seg_len: int = 32768, mode: str = "nondet") -> Workload:
    """4096 x 32768 float64 uniform in [-1e6, 1e6] with 1% of entries replaced by
    one of +inf, -inf, +0.0, -0.0 (uniformly); k=256, max, keys only. Mode
    "nondet": not_guaranteed + unspecified + unsorted; mode "det": gpu_to_gpu +
    unspecified + stable_sorted."""
    g = _rng(1005)
    n = segments * seg_len
    x = g.uniform(-1e6, 1e6, size=n)
    sp = g.random(n) < 0.01
    which = g.integers(0, 4, size=n)
    special = np.array([np.inf, -np.inf, 0.0, -0.0])
    x[sp] = special[which[sp]]
    if mode == "det":
        det, tie, order = "gpu_to_gpu", "unspecified", "stable_sorted"
    else:
        det, tie, order = "not_guaranteed", "unspecified", "unsorted"
    return Workload("f64 %d x %d with +/-inf +/-0, k=256 max keys (%s)" % (segments, seg_len, mode),
                    "f64", f64_bits(x), None, offsets_from_lengths([seg_len] * segments), 256,
                    "max", det, tie, order)


def array_workload(n: int = 1 << 28) -> Workload:
    """Top-k over one array (no segments): 2^28 fp32 keys ~ N(0,1), k=1024,
    max, pairs with value = int32 position, gpu_to_gpu + prefer_smaller_index
    + stable_sorted (one segment covering the whole array)."""
    g = _rng(1010)
    x = g.standard_normal(size=n, dtype=np.float32)
    return Workload("fp32 array of %d N(0,1), k=1024 max pairs (no segments)" % n, "f32", f32_bits(x),
                    np.arange(n, dtype=np.int32), offsets_from_lengths([n]), 1024, "max", "gpu_to_gpu",
                    "prefer_smaller_index", "stable_sorted", info={"array": True})


def by_number(cfg: int, **kw) -> Workload:
    return {1: workload1, 2: workload2, 3: workload3, 4: workload4, 5: workload5}[cfg](**kw)


# --------------------------------------------------------------------------
# Generic generators for parity and edge-case tests
# --------------------------------------------------------------------------

def random_keys(g: np.random.Generator, dtype: str, n: int, distinct: int | None = None,
                specials: bool = True) -> np.ndarray:
    """Random raw key bits of `dtype`. With `distinct`, keys are drawn from that
    many levels (heavy ties). With `specials`, +/-0 and +/-inf (floats) or the
    extreme integers are mixed in."""
    if dtype in ("f16", "bf16", "f32", "f64"):
        if distinct:
            lv = g.uniform(-4, 4, size=distinct)
            x = lv[g.integers(0, distinct, size=n)]
        else:
            x = g.standard_normal(n) * 100.0
        x = x.astype(np.float64)
        if specials and n:
            sp = g.random(n) < 0.05
            vals = np.array([0.0, -0.0, np.inf, -np.inf])
            x[sp] = vals[g.integers(0, 4, size=int(sp.sum()))]
        if dtype == "f16":
            return f16_bits(x.astype(np.float16))
        if dtype == "bf16":
            return bf16_bits(x.astype(np.float32))
        if dtype == "f32":
            return f32_bits(x.astype(np.float32))
        return f64_bits(x)
    if dtype == "u32":
        if distinct:
            lv = g.integers(0, 2**32, size=distinct, dtype=np.uint64)
            r = lv[g.integers(0, distinct, size=n)]
        else:
            r = g.integers(0, 2**32, size=n, dtype=np.uint64)
        r = r.astype(np.uint32)
        if specials and n:
            sp = g.random(n) < 0.02
            r[sp] = np.array([0, 0xFFFFFFFF], dtype=np.uint32)[g.integers(0, 2, size=int(sp.sum()))]
        return r
    if dtype == "i32":
        if distinct:
            lv = g.integers(-2**31, 2**31, size=distinct, dtype=np.int64)
            r = lv[g.integers(0, distinct, size=n)]
        else:
            r = g.integers(-2**31, 2**31, size=n, dtype=np.int64)
        r = r.astype(np.int32)
        if specials and n:
            sp = g.random(n) < 0.02
            r[sp] = np.array([-2**31, 2**31 - 1, 0, -1], dtype=np.int32)[
                g.integers(0, 4, size=int(sp.sum()))]
        return r
    raise ValueError(dtype)


def random_workload(seed: int, dtype: str, lengths, k: int, direction: str = "max",
                    determinism: str = "gpu_to_gpu", tie_break: str = "prefer_smaller_index",
                    ordering: str = "stable_sorted", pairs: bool = True,
                    distinct: int | None = None, specials: bool = True,
                    lead: int = 0) -> Workload:
    """A workload with the given segment lengths. `lead` unused keys are put in
    front of the first segment so that segment starts are not 16-byte aligned."""
    g = _rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    n = int(lengths.sum()) + lead
    keys = random_keys(g, dtype, n, distinct=distinct, specials=specials)
    vals = g.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32) if pairs else None
    offs = offsets_from_lengths(lengths) + lead
    return Workload("random %s" % dtype, dtype, keys, vals, offs, k, direction, determinism,
                    tie_break, ordering)
