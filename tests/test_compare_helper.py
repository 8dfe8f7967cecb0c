"""The GPU parity comparison must reject wrong answers (checked on the CPU with
oracle outputs standing in for a GPU result)."""
import numpy as np
import pytest

from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import compare, run_oracle


@pytest.mark.parametrize("ordering", ["stable_sorted", "unsorted"])
def test_compare_rejects_planted_errors(ordering):
    wl = W.random_workload(8, "f32", [5, 40, 3000, 0, 70], 16, ordering=ordering, distinct=9)
    want_k, want_v = run_oracle(wl)
    compare(wl, want_k.copy(), want_v.copy(), want_k, want_v)  # identical passes
    S, k = wl.num_segments, wl.k
    cases = []
    gk = want_k.copy(); gk[2 * k + 3] ^= 1; cases.append((gk, want_v.copy()))      # key bit flipped
    gv = want_v.copy(); gv[1 * k + 0] += 1; cases.append((want_k.copy(), gv))     # value changed
    gk = want_k.copy(); gk[4] = 0; cases.append((gk, want_v.copy()))               # write past n (seg 0 has 5)
    gk = want_k.copy(); gk[0 * k + 5] = 7; cases.append((gk, want_v.copy()))       # tail slot touched
    if ordering == "unsorted":
        # a different element with the same multiset of keys but another value
        gv = want_v.copy(); gv[2 * k + 1], gv[2 * k + 2] = gv[2 * k + 2] + 0, gv[2 * k + 2]
        gv[2 * k + 1] = -5; cases.append((want_k.copy(), gv))
    else:
        gk = want_k.copy(); gv = want_v.copy()
        gk[2 * k + 0], gk[2 * k + 1] = gk[2 * k + 1], gk[2 * k + 0]
        gv[2 * k + 0], gv[2 * k + 1] = gv[2 * k + 1], gv[2 * k + 0]
        cases.append((gk, gv))                                                     # order swapped
    for gk, gv in cases:
        with pytest.raises(AssertionError):
            compare(wl, gk, gv, want_k, want_v)


def test_sorted_mode_accepts_any_order_of_equal_keys():
    # sorted (not stable): equal keys -- +0.0 and -0.0 included -- in any order
    keys = W.f32_bits(np.array([1.0, 0.0, -0.0, 2.0, 0.0, 1.0, -3.0], dtype=np.float32))
    vals = np.arange(7, dtype=np.int32) * 10
    wl = W.Workload("sorted", "f32", keys, vals, np.array([0, 7], dtype=np.int64), 6, "max", "gpu_to_gpu",
                    "prefer_smaller_index", "sorted")
    want_k, want_v = run_oracle(wl)   # 2.0, 1.0@0, 1.0@5, 0.0@1, -0.0@2, 0.0@4
    gk, gv = want_k.copy(), want_v.copy()
    gk[[3, 4]] = gk[[4, 3]]; gv[[3, 4]] = gv[[4, 3]]   # -0.0 before +0.0: equal keys
    gv[[1, 2]] = gv[[2, 1]]                            # the two 1.0s swapped
    compare(wl, gk, gv, want_k, want_v)
    bad = want_k.copy(), want_v.copy()
    bad[0][[0, 1]] = bad[0][[1, 0]]; bad[1][[0, 1]] = bad[1][[1, 0]]   # 1.0 before 2.0
    with pytest.raises(AssertionError):
        compare(wl, *bad, want_k, want_v)
    gv = want_v.copy(); gv[1], gv[2] = gv[2], gv[2]   # a value repeated, one lost
    with pytest.raises(AssertionError):
        compare(wl, want_k.copy(), gv, want_k, want_v)


def test_not_guaranteed_mode_accepts_any_boundary_ties():
    # keys 5, 3, 3, 3, 1 with k = 3: any two of the three 3s
    keys = np.array([5, 3, 3, 3, 1], dtype=np.uint32)
    vals = np.array([50, 31, 32, 33, 10], dtype=np.int32)
    wl = W.Workload("nondet", "u32", keys, vals, np.array([0, 5], dtype=np.int64), 3, "max",
                    "not_guaranteed", "unspecified", "unsorted")
    want_k, want_v = run_oracle(wl)   # 5@0, 3@1, 3@2
    compare(wl, np.array([3, 5, 3], dtype=np.uint32), np.array([33, 50, 31], dtype=np.int32),
            want_k, want_v)  # order free, another tie taken: valid
    for gk, gv in [(want_k.copy(), np.array([50, 31, 31], dtype=np.int32)),      # one element twice
                   (want_k.copy(), np.array([50, 31, 34], dtype=np.int32)),      # not an element
                   (np.array([5, 3, 1], dtype=np.uint32), np.array([50, 31, 10], dtype=np.int32))]:  # wrong keys
        with pytest.raises(AssertionError):
            compare(wl, gk, gv, want_k, want_v)
