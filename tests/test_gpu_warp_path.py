"""GPU parity of the warp-select paths (k <= 32: one warp per segment, or a
team of eight warps per segment sharing a bound) against the CPU oracle,
bit-exact: every key type, direction, tie-break and ordering on ragged
segments; segments shorter than, equal to and just above k; long segments
forced through either path (many queue merges, adversarial orders, heavy
ties); a batch split over all three paths; and the one key whose composite
equals an empty slot's."""
import itertools

import numpy as np
import pytest

import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import check_workload

pytestmark = pytest.mark.gpu

DTYPES = ["f16", "bf16", "f32", "f64", "u32", "i32"]
TIES = ["unspecified", "prefer_smaller_index", "prefer_larger_index"]
ORDERINGS = ["unsorted", "sorted", "stable_sorted"]
BIG = 1 << 20
# options that send every segment (up to BIG keys) through one path
PATHS = {"warp": dict(small_segment_max_len=BIG, team_segment_max_len=-1),
         "team": dict(small_segment_max_len=-1, team_segment_max_len=BIG)}
SHORT = [0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 100, 255, 256, 257, 1000, 2047, 2048,
         2049, 4095, 4096]


def det_for(tie, i):
    if tie != "unspecified":
        return "gpu_to_gpu"
    return ["not_guaranteed", "run_to_run", "gpu_to_gpu"][i % 3]


@pytest.mark.parametrize("path", ["warp", "team"])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("direction", ["max", "min"])
@pytest.mark.parametrize("tie", TIES)
def test_short_segment_matrix(path, dtype, direction, tie):
    for i, (k, distinct) in enumerate([(1, None), (7, 5), (16, None), (32, 40), (32, None)]):
        ordering = ORDERINGS[i % 3]
        wl = W.random_workload(300 + i, dtype, SHORT, k, direction, det_for(tie, i), tie, ordering,
                               pairs=(i % 2 == 0), distinct=distinct, lead=i)
        check_workload(wl, **PATHS[path], where="%s %s/%s/%s k=%d %s" % (path, dtype, direction, tie, k, ordering))
        assert st.last_launch_count() == 1  # every segment took that path


@pytest.mark.parametrize("path", ["warp", "team"])
@pytest.mark.parametrize("dtype", ["f16", "f32", "f64", "u32"])
def test_every_length_up_to_k_plus_a_few(path, dtype):
    lengths = list(range(0, 41))
    for k, tie, ordering in itertools.product([1, 2, 31, 32], ["prefer_smaller_index", "prefer_larger_index"],
                                              ["unsorted", "stable_sorted"]):
        wl = W.random_workload(11 + k, dtype, lengths, k, "max" if k % 2 else "min", "gpu_to_gpu", tie,
                               ordering, pairs=True, distinct=6, lead=k % 5)
        check_workload(wl, **PATHS[path], where="%s lengths 0..40 %s k=%d %s %s" % (path, dtype, k, tie, ordering))


@pytest.mark.parametrize("dtype", ["f16", "f32", "f64", "u32"])
def test_mixed_warp_team_and_cta_segments(dtype):
    """Short segments take single warps, middle ones teams, long ones CTAs:
    three launches, one result."""
    lengths = [0, 5, 4096, 4097, 3000, 70000, 12, 20000, 4095, 150000, 1]
    for i, (k, tie, ordering) in enumerate([(8, "prefer_smaller_index", "stable_sorted"),
                                            (32, "prefer_larger_index", "unsorted"),
                                            (20, "prefer_larger_index", "sorted")]):
        wl = W.random_workload(40 + i, dtype, lengths, k, "max" if i % 2 == 0 else "min", "gpu_to_gpu", tie,
                               ordering, pairs=True, distinct=(None if i == 0 else 30), lead=2)
        check_workload(wl, small_segment_max_len=1024, team_segment_max_len=8192,
                       where="mixed %s k=%d %s %s" % (dtype, k, tie, ordering))
        assert st.last_launch_count() == 3


@pytest.mark.parametrize("path", ["warp", "team"])
@pytest.mark.parametrize("dtype", ["f16", "f32", "f64", "i32"])
def test_long_segments_forced_through_warps(path, dtype):
    lengths = [40001, 131072, 7, 65536 + 3]
    for i, (k, tie, ordering, distinct) in enumerate([(32, "prefer_smaller_index", "stable_sorted", None),
                                                      (9, "prefer_larger_index", "sorted", 3),
                                                      (32, "prefer_larger_index", "unsorted", 1000)]):
        wl = W.random_workload(70 + i, dtype, lengths, k, "min" if i % 2 else "max", "gpu_to_gpu", tie, ordering,
                               pairs=True, distinct=distinct, lead=1)
        check_workload(wl, **PATHS[path], where="forced %s %s k=%d %s %s" % (path, dtype, k, tie, ordering))
        assert st.last_launch_count() == 1


@pytest.mark.parametrize("path", ["warp", "team"])
@pytest.mark.parametrize("pattern", ["ascending", "descending", "all_equal", "sawtooth"])
def test_orders_that_flush_the_queue_often(path, pattern):
    n = 50000
    i = np.arange(n, dtype=np.int64)
    x = {"ascending": i, "descending": n - i, "all_equal": np.full(n, 77), "sawtooth": i % 97}[pattern]
    x = x.astype(np.uint32)
    for direction, tie, k in itertools.product(["max", "min"], ["prefer_smaller_index", "prefer_larger_index"],
                                               [1, 32]):
        wl = W.Workload(pattern, "u32", x, i.astype(np.int32), W.offsets_from_lengths([n // 2, n // 2]), k,
                        direction, "gpu_to_gpu", tie, "stable_sorted")
        check_workload(wl, **PATHS[path], where="%s %s %s %s k=%d" % (path, pattern, direction, tie, k))


@pytest.mark.parametrize("path", ["warp", "team"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "f64"])
def test_signed_zeros_and_infinities_short(path, dtype):
    g = np.random.Generator(np.random.PCG64(19))
    x = g.choice(np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0]), size=6000, p=[.3, .3, .05, .05, .15, .15])
    bits = {"f16": W.f16_bits, "f32": W.f32_bits, "f64": W.f64_bits}[dtype](x)
    offs = W.offsets_from_lengths([3, 17, 40, 1000, 4000])
    for direction, tie, k in itertools.product(["max", "min"], TIES[1:], [3, 32]):
        wl = W.Workload("zeros", dtype, bits[: offs[-1]], np.arange(offs[-1], dtype=np.int32), offs, k,
                        direction, "gpu_to_gpu", tie, "stable_sorted")
        check_workload(wl, **PATHS[path], where="%s zeros %s %s %s k=%d" % (path, dtype, direction, tie, k))


@pytest.mark.parametrize("path", ["warp", "team"])
def test_key_equal_to_an_empty_slot(path):
    """u32 key 0xFFFFFFFF under min (rank all ones) at source index 0 with
    larger indices preferred: its composite equals an empty slot's."""
    for direction, worst in (("min", 0xFFFFFFFF), ("max", 0)):
        for n, k in ((1, 1), (3, 5), (5, 5), (6, 5), (32, 32), (40, 32)):
            x = np.arange(100, 100 + n, dtype=np.uint32)
            x[0] = worst
            if n > 2:
                x[2] = worst
            for ordering in ORDERINGS:
                wl = W.Workload("empty-slot", "u32", x, np.arange(n, dtype=np.int32) * 3,
                                np.array([0, n], dtype=np.int64), k, direction, "gpu_to_gpu",
                                "prefer_larger_index", ordering)
                check_workload(wl, **PATHS[path], where="%s empty slot %s n=%d k=%d %s" % (
                    path, direction, n, k, ordering))


@pytest.mark.parametrize("path", ["warp", "team"])
def test_offsets_edge_cases_warp_path(path):
    g = np.random.Generator(np.random.PCG64(3))
    keys = W.random_keys(g, "f32", 5000)
    vals = np.arange(5000, dtype=np.int32)
    offs = np.array([0, 10, 4, 4, 20, 60, 61, 61, 4000, 3000, 5000], dtype=np.int64)
    for k in (1, 10, 32):
        for order in ORDERINGS:
            wl = W.Workload("edges", "f32", keys, vals, offs, k, "max", "gpu_to_gpu", "prefer_smaller_index", order)
            check_workload(wl, **PATHS[path], where="%s edges k=%d %s" % (path, k, order))
            check_workload(wl, **PATHS[path], max_segment_len=None, where="%s edges k=%d %s unknown len" % (
                path, k, order))


def test_automatic_choice():
    """Automatic mode: with at least one segment per SM, segments up to 4096
    keys take single warps and longer ones CTAs (two launches); a few short
    segments take one team launch; k > 32 takes CTAs."""
    g = np.random.Generator(np.random.PCG64(5))
    lengths = list(g.integers(0, 3000, size=400)) + [30000]
    wl = W.random_workload(61, "f32", lengths, 16, "max", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted",
                           pairs=True, lead=1)
    check_workload(wl, where="auto many")
    assert st.last_launch_count() == 2
    wl = W.random_workload(62, "f32", lengths[:20], 16, "min", "gpu_to_gpu", "prefer_larger_index", "unsorted",
                           pairs=True, lead=1)
    check_workload(wl, where="auto few")
    assert st.last_launch_count() == 1
    wl = W.random_workload(63, "f32", lengths, 33, "max", "gpu_to_gpu", "prefer_smaller_index", "sorted",
                           pairs=False, lead=1)
    check_workload(wl, where="auto k=33")
    assert st.last_launch_count() == 1
