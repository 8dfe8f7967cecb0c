"""The bounded wait on a bulk copy, exercised on the GPU without a fault.

Every wait of the segment kernel on a ring stage gives up after a bound of
SM clock cycles, sets bit 0 of the device error word, stops the CTA (the
whole cluster, when one CTA stops) after letting copies in flight land, and
returns. The instrumented build (libsegtopk_instr.so) lets a test shorten
that bound and add bytes to the expected count of every slice's first copy,
so that its wait runs out while the copy itself completes: nothing hangs,
nothing traps, and the device stays usable.
"""
import numpy as np
import pytest

import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import SENTINEL_VALUE, check_workload, run_gpu

pytestmark = pytest.mark.gpu

SHORT_WAIT = 1 << 20       # about half a millisecond of SM clock cycles
DEFAULT_WAIT = 1 << 31


@pytest.fixture(scope="module")
def instr():
    L = st.load_instrumented()
    yield L
    st.set_test_hooks(DEFAULT_WAIT, 0)


def workload():
    # every segment has at least one ring chunk on every CTA of a 2-CTA cluster
    return W.random_workload(8100, "f32", [40000, 100000, 70001, 65536], 50, "max", "gpu_to_gpu",
                             "prefer_smaller_index", "stable_sorted", pairs=True, distinct=500, lead=1)


@pytest.mark.parametrize("width", [1, 2])
def test_wait_that_runs_out_sets_the_error_bit_and_returns(instr, width):
    wl = workload()
    # the instrumented build, hooks at their defaults, matches the oracle
    st.set_test_hooks(DEFAULT_WAIT, 0)
    check_workload(wl, cluster_width=width, lib=instr, where="instrumented build C=%d" % width)
    # every slice's first copy now never completes its expected byte count
    st.set_test_hooks(SHORT_WAIT, 16)
    try:
        got_k, got_v = run_gpu(wl, cluster_width=width, lib=instr)
        err = st.read_device_error(lib=instr)
    finally:
        st.set_test_hooks(DEFAULT_WAIT, 0)
    assert err & 1, "the copy wait did not report running out (error word %#x)" % err
    # the stopped segments wrote nothing: every output slot keeps its fill
    assert np.all(got_v == SENTINEL_VALUE)
    # the context is still usable: the same call now matches the oracle
    check_workload(wl, cluster_width=width, lib=instr, where="after the bounded wait C=%d" % width)


def test_statistics_counters(instr):
    st.set_test_hooks(DEFAULT_WAIT, 0)
    st.read_stats()  # clear
    wl = workload()
    check_workload(wl, cluster_width=1, lib=instr)
    s = st.read_stats()
    assert s["ctas"] == wl.num_segments
    assert s["keys"] == int(wl.lengths.sum())
    assert s["chunks"] > 0 and s["cycles"] > 0 and s["digit_passes"] > 0
    assert s["list_entries"] >= min(wl.k, int(wl.lengths.min())) * wl.num_segments
