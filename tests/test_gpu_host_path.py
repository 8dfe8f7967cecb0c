"""GPU parity of the host-buffer entry points against the CPU oracle.

segtopk_batched_topk_host (caller's device workspace) and
segtopk_batched_topk_host_noalloc (the library's fixed staging array) take
host arrays: they copy keys and offsets to the device, select there, and
gather the selected values from the host array by the source indices the
kernel returns. Both are compared slot by slot with the oracle on the same
seeded inputs, with the output pre-filled by a sentinel that slots past a
short segment's length must keep ("Top-K: Determinism, Tie-Breaking, and
Output Ordering", "Which items are selected?" and "Output ordering").
"""
import numpy as np
import pytest
import torch

import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import (NUMPY_SIGNED, SENTINEL_BITS, SENTINEL_VALUE, TORCH_VIEW, compare, run_oracle)

pytestmark = pytest.mark.gpu


def run_host(wl, noalloc: bool, pinned: bool = True):
    """(out key bits, out values) of a host-buffer entry point, as numpy."""
    kb = W.KEY_BYTES[wl.dtype]
    keys = torch.from_numpy(np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype]).copy())
    offs = torch.from_numpy(wl.offsets.copy())
    vals = torch.from_numpy(wl.values.copy()) if wl.values is not None else None
    S, k = wl.num_segments, wl.k
    sent = np.array([SENTINEL_BITS[kb]], dtype=np.uint64).astype(
        {2: np.uint16, 4: np.uint32, 8: np.uint64}[kb]).view(NUMPY_SIGNED[wl.dtype])[0]
    out_k = torch.full((S * k,), int(sent), dtype=TORCH_VIEW[wl.dtype])
    out_v = torch.full((S * k,), SENTINEL_VALUE, dtype=torch.int32) if vals is not None else None
    if pinned:
        keys, offs, out_k = keys.pin_memory(), offs.pin_memory(), out_k.pin_memory()
        vals = vals.pin_memory() if vals is not None else None
        out_v = out_v.pin_memory() if out_v is not None else None
    args = dict(values=vals, direction=wl.direction, determinism=wl.determinism, tie_break=wl.tie_break,
                ordering=wl.ordering, out_keys=out_k, out_values=out_v, max_segment_len=wl.max_segment_len)
    if noalloc:
        st.batched_topk_host_noalloc(wl.dtype, keys, offs, k, **args)
    else:
        ws = st.host_workspace_bytes(wl.dtype, vals is not None, wl.num_keys, S, k)
        workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
        st.batched_topk_host(wl.dtype, keys, offs, k, workspace, **args)
    assert st.read_device_error() == 0
    gk = out_k.numpy().view(W.STORAGE[wl.dtype] if wl.dtype != "i32" else np.uint32)
    if wl.dtype == "i32":
        gk = gk.view(np.int32)
    return gk.copy(), (out_v.numpy().copy() if out_v is not None else None)


# ragged: empty, shorter than k (sentinel tails), around vector and chunk
# boundaries, several chunks; `lead` unused keys put every segment start off
# a 16-byte boundary
CASES = [
    ("f32", [0, 1, 3, 49, 50, 51, 1000, 4097, 20000, 70001], 50, "max", "gpu_to_gpu",
     "prefer_smaller_index", "stable_sorted", True, 300, 3),
    ("f16", [5, 0, 31, 32, 33, 900, 5000, 16385, 40000], 32, "min", "gpu_to_gpu", "prefer_larger_index",
     "unsorted", True, 40, 1),
    ("f64", [2, 7, 8, 9, 256, 1500, 9000, 33000], 8, "max", "not_guaranteed", "unspecified", "unsorted",
     False, None, 1),
    ("u32", [0, 1024, 1023, 1025, 65536, 100000], 1024, "max", "gpu_to_gpu", "prefer_smaller_index", "sorted",
     True, 17, 2),
    ("bf16", [3, 64, 129, 3000], 100, "min", "run_to_run", "unspecified", "stable_sorted", True, 9, 5),
    ("i32", [1, 2, 70000, 0, 12], 7, "max", "gpu_to_gpu", "prefer_larger_index", "stable_sorted", False, 50, 3),
]


@pytest.mark.parametrize("noalloc", [False, True], ids=["workspace", "noalloc"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_entry_points_match_the_oracle(case, noalloc):
    dtype, lengths, k, direction, det, tie, ordering, pairs, distinct, lead = case
    wl = W.random_workload(4000 + len(lengths), dtype, lengths, k, direction, det, tie, ordering, pairs=pairs,
                           distinct=distinct, lead=lead)
    got_k, got_v = run_host(wl, noalloc)
    want_k, want_v = run_oracle(wl)
    compare(wl, got_k, got_v, want_k, want_v, where="%s host (%s)" % (dtype, "noalloc" if noalloc else "workspace"))


@pytest.mark.parametrize("noalloc", [False, True], ids=["workspace", "noalloc"])
def test_host_entry_points_on_workload_shapes(noalloc):
    # workload 1 as benchmarked, and workload 2's shape (logit rows, value =
    # source index) shortened to fit the no-allocation staging array
    for wl in (W.workload1(), W.workload2(segments=24, seg_len=152064)):
        got_k, got_v = run_host(wl, noalloc)
        want_k, want_v = run_oracle(wl)
        compare(wl, got_k, got_v, want_k, want_v, where=wl.name)


def test_host_entry_point_with_pageable_buffers():
    wl = W.random_workload(4100, "f32", [17, 3000, 9], 16, "min", "gpu_to_gpu", "prefer_smaller_index",
                           "stable_sorted", pairs=True, distinct=30, lead=1)
    got_k, got_v = run_host(wl, noalloc=False, pinned=False)
    want_k, want_v = run_oracle(wl)
    compare(wl, got_k, got_v, want_k, want_v, where="pageable host buffers")
