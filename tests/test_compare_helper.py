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
