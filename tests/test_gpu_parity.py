"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
bit-exact, on seeded inputs that span several 32 KiB chunks, ragged tails,
unaligned segment starts, single CTAs and forced thread-block clusters."""
import itertools

import numpy as np
import pytest

from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import check_workload, run_gpu

pytestmark = pytest.mark.gpu

DTYPES = ["f16", "bf16", "f32", "f64", "u32", "i32"]
TIES = ["unspecified", "prefer_smaller_index", "prefer_larger_index"]
ORDERINGS = ["unsorted", "sorted", "stable_sorted"]
# ragged lengths: empty, tiny, around vector / chunk boundaries, several chunks
LENGTHS = [0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 100, 1000, 2047, 2048, 2049, 4095, 4096, 4097,
           8191, 8193, 12000, 20000, 40001]


def det_for(tie, i):
    if tie != "unspecified":
        return "gpu_to_gpu"
    return ["not_guaranteed", "run_to_run", "gpu_to_gpu"][i % 3]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("direction", ["max", "min"])
@pytest.mark.parametrize("tie", TIES)
def test_single_cta_matrix(dtype, direction, tie):
    for i, (k, distinct) in enumerate([(1, None), (7, 5), (50, None), (300, 40), (2048, None)]):
        ordering = ORDERINGS[i % 3]
        wl = W.random_workload(100 + i, dtype, LENGTHS, k, direction, det_for(tie, i), tie, ordering,
                               pairs=(i % 2 == 0), distinct=distinct, lead=1 + i)
        check_workload(wl, cluster_width=1, where="%s/%s/%s k=%d %s" % (dtype, direction, tie, k, ordering))


@pytest.mark.parametrize("width", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["f16", "f32", "f64", "u32"])
def test_cluster_widths(width, dtype):
    lengths = [0, 1, 3, width - 1, width, 17, 100, 4097, 30000, 70001, 131072]
    for i, (k, tie, ordering, distinct) in enumerate([
            (5, "prefer_smaller_index", "stable_sorted", None),
            (64, "prefer_larger_index", "unsorted", 7),
            (1024, "prefer_smaller_index", "sorted", 300),
            (33, "prefer_larger_index", "stable_sorted", 3)]):
        direction = "max" if i % 2 == 0 else "min"
        wl = W.random_workload(500 + i, dtype, lengths, k, direction, "gpu_to_gpu", tie, ordering,
                               pairs=True, distinct=distinct, lead=3)
        check_workload(wl, cluster_width=width, where="C=%d %s k=%d %s %s" % (width, dtype, k, tie, ordering))


@pytest.mark.parametrize("dtype", ["f32", "f16", "f64"])
def test_signed_zero_and_infinities(dtype):
    """Only +/-0.0, +/-inf and a few numbers: zeros tie and keep their bits."""
    g = np.random.Generator(np.random.PCG64(9))
    n = 30000
    x = g.choice(np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0]), size=n, p=[.3, .3, .05, .05, .15, .15])
    bits = {"f16": W.f16_bits, "f32": W.f32_bits, "f64": W.f64_bits}[dtype](x)
    lengths = [17, 1000, 9000, 19983]
    offs = W.offsets_from_lengths(lengths)
    for direction, tie, k in itertools.product(["max", "min"], TIES[1:], [3, 700, 2048]):
        wl = W.Workload("zeros", dtype, bits[: offs[-1]], np.arange(offs[-1], dtype=np.int32), offs, k,
                        direction, "gpu_to_gpu", tie, "stable_sorted")
        for width in (1, 2):
            check_workload(wl, cluster_width=width, where="zeros %s %s %s k=%d C=%d" % (
                dtype, direction, tie, k, width))


def test_nan_order_reading():
    """NaNs (pages silent): +NaN above +inf and -NaN below -inf, payload order."""
    bits = np.array([0x7F800000, 0x7FC00001, 0xFF800000, 0xFFC00100, 0x7FC00100, 0xFFC00001, 0,
                     0x3F800000] * 700, dtype=np.uint32)
    offs = np.array([0, 5, 5600], dtype=np.int64)
    for direction in ("max", "min"):
        wl = W.Workload("nan", "f32", bits, np.arange(len(bits), dtype=np.int32), offs, 9, direction,
                        "gpu_to_gpu", "prefer_smaller_index", "stable_sorted")
        check_workload(wl, cluster_width=1)
        check_workload(wl, cluster_width=2)


@pytest.mark.parametrize("pattern", ["ascending", "descending", "all_equal", "two_values", "sawtooth"])
@pytest.mark.parametrize("tie", ["prefer_smaller_index", "prefer_larger_index"])
def test_adversarial_orders(pattern, tie):
    """Orders that make the candidate list refill and trim repeatedly."""
    n = 200000
    i = np.arange(n, dtype=np.int64)
    if pattern == "ascending":
        x = i.astype(np.uint32)
    elif pattern == "descending":
        x = (n - i).astype(np.uint32)
    elif pattern == "all_equal":
        x = np.full(n, 77, dtype=np.uint32)
    elif pattern == "two_values":
        x = np.where(i % 3 == 0, 5, 9).astype(np.uint32)
    else:
        x = (i % 5000).astype(np.uint32)
    lengths = [n // 2, n // 4, n // 4]
    for direction, k in itertools.product(["max", "min"], [1, 100, 1500]):
        wl = W.Workload(pattern, "u32", x, i.astype(np.int32), W.offsets_from_lengths(lengths), k,
                        direction, "gpu_to_gpu", tie, "stable_sorted")
        for width in (1, 4):
            check_workload(wl, cluster_width=width, where="%s %s %s k=%d C=%d" % (
                pattern, tie, direction, k, width))


@pytest.mark.parametrize("tie", ["prefer_smaller_index", "prefer_larger_index"])
def test_f64_bounds_on_either_side_of_zero(tie):
    """f64 keys whose bound lies below +0.0 for max or at or above it for
    min (the candidate test's general path), and ordered runs across zero
    whose bound changes sign during the stream."""
    g = np.random.Generator(np.random.PCG64(3100))
    n = 70000
    neg = -np.abs(g.standard_normal(n) * 50.0) - 1e-3         # all negative
    pos = np.abs(g.standard_normal(n) * 50.0)                 # all non-negative, with ties at +0.0
    pos[::997] = 0.0
    pos[::1009] = -0.0
    ramp = np.linspace(-1000.0, 1000.0, n)                     # ascending through zero
    x = np.concatenate([neg, pos, ramp, ramp[::-1], neg[:5000] * 1e-300]).astype(np.float64)
    lengths = [n, n, n, n, 5000]
    i = np.arange(x.size, dtype=np.int32)
    for direction, k in itertools.product(["max", "min"], [1, 50, 700]):
        wl = W.Workload("f64 signs", "f64", W.f64_bits(x), i, W.offsets_from_lengths(lengths), k,
                        direction, "gpu_to_gpu", tie, "stable_sorted")
        for width in (1, 3):
            check_workload(wl, cluster_width=width, where="f64 signs %s %s k=%d C=%d" % (tie, direction, k, width))


def test_offsets_edge_cases():
    """Decreasing offsets (empty), a zero-length batch of segments, n == k,
    n == k + 1, every segment shorter than k."""
    g = np.random.Generator(np.random.PCG64(3))
    keys = W.random_keys(g, "f32", 5000)
    vals = np.arange(5000, dtype=np.int32)
    offs = np.array([0, 10, 4, 4, 20, 60, 61, 61, 4000, 3000, 5000], dtype=np.int64)
    for k in (1, 10, 40, 41, 2048):
        for order in ORDERINGS:
            wl = W.Workload("edges", "f32", keys, vals, offs, k, "max", "gpu_to_gpu",
                            "prefer_smaller_index", order)
            check_workload(wl, cluster_width=1, where="edges k=%d %s" % (k, order))
            check_workload(wl, cluster_width=3, where="edges k=%d %s C=3" % (k, order))


def test_unknown_max_segment_len():
    wl = W.random_workload(4, "f32", [10, 5000, 300], 20, pairs=True, lead=5)
    check_workload(wl, max_segment_len=None)


def _segment_sets(wl, out_k, out_v):
    k = wl.k
    m = np.minimum(wl.lengths, k)
    return [sorted(zip(out_k[s * k: s * k + m[s]].tolist(), out_v[s * k: s * k + m[s]].tolist()))
            for s in range(wl.num_segments)]


def test_repeat_runs_identical():
    """Deterministic modes: the selected set is identical run after run
    (unsorted positions may move); sorted outputs are bit-identical."""
    wl = W.workload3(segments=300)
    a = run_gpu(wl)
    sa = _segment_sets(wl, *a)
    for _ in range(3):
        assert _segment_sets(wl, *run_gpu(wl)) == sa
    wl = W.workload4(segments=3)
    a = run_gpu(wl)
    for _ in range(2):
        b = run_gpu(wl)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("dtype", ["f32", "f64", "f16", "u32"])
def test_many_single_cta_segments(dtype):
    """Several waves of single-CTA segments (more segments than resident
    CTAs), the sample size of the speculative bound chosen for many waves.
    Lengths mix empty, tiny, n <= k and multi-chunk segments at unaligned
    starts."""
    g = np.random.Generator(np.random.PCG64(77))
    lengths = np.where(g.random(1400) < 0.1, 0, g.integers(1, 20000, size=1400))
    lengths[::37] = g.integers(20000, 60000, size=len(lengths[::37]))
    for i, (k, tie, ordering, direction) in enumerate([
            (1, "prefer_smaller_index", "stable_sorted", "max"),
            (50, "prefer_larger_index", "unsorted", "min"),
            (300, "prefer_smaller_index", "sorted", "max"),
            (2048, "prefer_larger_index", "stable_sorted", "min")]):
        wl = W.random_workload(900 + i, dtype, lengths, k, direction, "gpu_to_gpu", tie, ordering,
                               pairs=(i % 2 == 0), distinct=(40 if i == 1 else None), lead=1 + i)
        check_workload(wl, cluster_width=1, where="many segments %s k=%d %s %s" % (dtype, k, tie, ordering))


@pytest.mark.parametrize("dtype", ["f16", "f32", "f64", "u32"])
def test_offset_view_of_the_key_array(dtype):
    """keys[1:] of a device array: the key pointer is aligned to its element
    size only, so no segment starts on a 16-byte boundary of the pointer's
    own array; every path (single warp, team, CTA, cluster) reads it."""
    from tests.gpu_util import to_device_keys
    lengths = [0, 1, 5, 31, 33, 700, 4095, 9000, 40001, 150000]
    for i, (k, width, small, team) in enumerate([(8, 0, 0, 0), (32, 1, -1, -1), (300, 0, 0, 0),
                                                 (50, 3, -1, -1), (16, 0, 100000, -1), (24, 0, -1, 100000)]):
        full = W.random_workload(900 + i, dtype, lengths, k, "max" if i % 2 else "min", "gpu_to_gpu",
                                 ["prefer_smaller_index", "prefer_larger_index"][i % 2],
                                 ["stable_sorted", "unsorted"][i % 2], pairs=True, distinct=200, lead=1)
        wl = W.Workload("view", dtype, full.keys[1:], full.values[1:], full.offsets - 1, k, full.direction,
                        full.determinism, full.tie_break, full.ordering)
        keys_full = to_device_keys(full)
        view = keys_full[1:]
        assert view.data_ptr() % 16 != 0
        check_workload(wl, cluster_width=width, keys_t=view, small_segment_max_len=small,
                       team_segment_max_len=team, where="%s view k=%d C=%d" % (dtype, k, width))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32", "f64", "u32", "i32"])
def test_too_small_length_hint_is_reported(dtype):
    """A max_segment_len hint below the longest segment is a caller error:
    the longer segments are left unwritten and bit 1 of the device error word
    is set, read back per key type (every kernel translation unit has its
    own word); the other segments are still exact."""
    import segmented_radix_top_gb300 as st
    from tests.gpu_util import SENTINEL_VALUE, compare, run_oracle
    lengths = [10, 3000, 9000, 60000, 100]
    for k, width in [(8, 0), (50, 1), (50, 2)]:
        wl = W.random_workload(950 + k + width, dtype, lengths, k, "max", "gpu_to_gpu", "prefer_smaller_index",
                               "stable_sorted", pairs=True, distinct=100, lead=1)
        assert st.read_device_error() == 0
        got_k, got_v = run_gpu(wl, cluster_width=width, max_segment_len=9000)
        err = st.read_device_error()
        assert err == 2, "error word %#x (want the segment-too-long bit)" % err
        v = got_v.reshape(wl.num_segments, k)
        assert np.all(v[3] == SENTINEL_VALUE)  # the 60000-key segment is left unwritten
        keep = np.array([0, 1, 2, 4])
        sub = W.Workload("hint", dtype, wl.keys, wl.values, wl.offsets, k, wl.direction, wl.determinism,
                         wl.tie_break, wl.ordering)
        want_k, want_v = run_oracle(sub)
        gk, wk = got_k.reshape(-1, k)[keep].reshape(-1), want_k.reshape(-1, k)[keep].reshape(-1)
        gv, wv = v[keep].reshape(-1), want_v.reshape(-1, k)[keep].reshape(-1)
        offs = np.concatenate([[0], np.cumsum(np.array(lengths)[keep])])
        part = W.Workload("hint", dtype, np.zeros(int(offs[-1]), dtype=wl.keys.dtype), None, offs, k,
                          wl.direction, wl.determinism, wl.tie_break, wl.ordering)
        compare(part, gk, gv, wk, wv, where="%s k=%d C=%d short segments" % (dtype, k, width))


@pytest.mark.parametrize("width", [1, 4])
def test_not_guaranteed_ties_and_unstable_sort(width):
    """The cheaper variants: not_guaranteed takes surplus boundary ties in any
    order (no selection by index), sorted without stability sorts 64-bit
    keys on the key alone. Half of every long segment ties at one value
    (the k-th key falls inside the tie block), as in the u32 workload;
    checked by the contract of each mode (multisets, order, real elements)."""
    g = np.random.Generator(np.random.PCG64(960 + width))
    lengths = [7, 300, 5000, 70001, 131072]
    n = sum(lengths)
    keys = g.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    keys[g.random(n) < 0.5] = 0xFFC00000
    offs = W.offsets_from_lengths(lengths)
    vals = g.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32)
    for k, ordering in [(1024, "unsorted"), (1024, "sorted"), (100, "stable_sorted"), (600, "unsorted")]:
        wl = W.Workload("ties", "u32", keys, vals, offs, k, "max", "not_guaranteed", "unspecified", ordering)
        check_workload(wl, cluster_width=width, where="u32 ties nondet k=%d %s C=%d" % (k, ordering, width))
    f = W.random_workload(970 + width, "f64", [600, 3000, 40000, 90001], 600, "max", "gpu_to_gpu",
                          "prefer_smaller_index", "sorted", pairs=True, distinct=50)
    check_workload(f, cluster_width=width, where="f64 sorted k=600 C=%d" % width)
    w = W.random_workload(980 + width, "f16", [33, 500, 4000, 9000], 24, "min", "gpu_to_gpu",
                          "prefer_larger_index", "sorted", pairs=True, distinct=12)
    check_workload(w, cluster_width=0, small_segment_max_len=100000, where="f16 warp sorted prefer_larger")
    check_workload(w, cluster_width=0, team_segment_max_len=100000, small_segment_max_len=-1,
                   where="f16 team sorted prefer_larger")
