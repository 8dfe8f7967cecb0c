"""The host-buffer entry point that allocates no device memory.

segtopk_batched_topk_host_noalloc is for callers that cannot allocate device
memory themselves: a plugin inside a program whose caching allocator owns the
GPU's memory, or code held to a fixed device-memory budget. It stages each
call in a fixed array inside the library instead of a workspace the caller
allocates. Its results must equal those of segtopk_batched_topk_host, the
entry point that takes the caller's workspace.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NUMPY_SIGNED = {"f16": np.int16, "f32": np.int32, "f64": np.int64, "u32": np.int32}
TORCH_VIEW = {"f16": torch.int16, "f32": torch.int32, "f64": torch.int64, "u32": torch.int32}


@pytest.fixture(scope="module", autouse=True)
def library():
    st.build()
    st.load()


def host_tensors(wl):
    keys = torch.from_numpy(np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype]).copy())
    offs = torch.from_numpy(wl.offsets.copy())
    vals = torch.from_numpy(wl.values.copy()) if wl.values is not None else None
    S, k = wl.num_segments, wl.k
    # a fill that slots past a short segment's length must keep
    out_k = torch.full((S * k,), 0x5A5A, dtype=TORCH_VIEW[wl.dtype])
    out_v = torch.full((S * k,), -123456789, dtype=torch.int32) if vals is not None else None
    return keys, offs, vals, out_k, out_v


def run_both(wl):
    """(no-alloc result, workspace result), each as (keys, values) numpy arrays."""
    keys, offs, vals, out_k, out_v = host_tensors(wl)
    args = dict(values=vals, direction=wl.direction, determinism=wl.determinism, tie_break=wl.tie_break,
                ordering=wl.ordering, max_segment_len=wl.max_segment_len)

    nk, nv = out_k.clone(), out_v.clone() if out_v is not None else None
    st.batched_topk_host_noalloc(wl.dtype, keys, offs, wl.k, out_keys=nk, out_values=nv, **args)

    ws_bytes = st.host_workspace_bytes(wl.dtype, vals is not None, wl.num_keys, wl.num_segments, wl.k)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rk, rv = out_k.clone(), out_v.clone() if out_v is not None else None
    st.batched_topk_host(wl.dtype, keys, offs, wl.k, workspace, out_keys=rk, out_values=rv, **args)
    torch.cuda.synchronize()
    assert st.read_device_error() == 0

    def np_of(t):
        return None if t is None else t.numpy().copy()
    return (np_of(nk), np_of(nv)), (np_of(rk), np_of(rv))


def assert_same(a, b, where):
    assert np.array_equal(a[0], b[0]), "%s: keys differ from the workspace entry point" % where
    if b[1] is not None:
        assert np.array_equal(a[1], b[1]), "%s: values differ from the workspace entry point" % where


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    # first call: f32 pairs, several chunks per segment, ragged and unaligned
    first = W.random_workload(7001, "f32", [0, 1, 5, 49, 50, 51, 1000, 4097, 20000, 65536, 131071], 50,
                              "max", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted", pairs=True,
                              distinct=300, lead=3)
    # second call: smaller, another key type and mode, segments shorter than k
    # (their tail slots must keep the caller's contents, not the first call's)
    second = W.random_workload(7002, "f64", [3, 0, 7, 8, 9, 300, 2048, 5000], 8, "min", "gpu_to_gpu",
                               "prefer_larger_index", "stable_sorted", pairs=True, distinct=20, lead=1)
    for i, wl in enumerate([first, second]):
        got, want = run_both(wl)
        assert_same(got, want, "call %d (%s)" % (i + 1, wl.name))


def test_workload_shape_keys_only_twice():
    # 16 ragged fp32 segments of up to 4096 keys, k = 8, keys only, twice in a row
    wl = W.workload1()
    a, ref = run_both(wl)
    assert_same(a, ref, "first call")
    b, _ = run_both(wl)
    assert_same(b, ref, "second call")


def test_request_beyond_the_staging_size_is_refused():
    n = st.NOALLOC_STAGING_BYTES // 4 + 1024  # fp32 keys alone exceed the staging array
    keys = torch.zeros(n, dtype=torch.int32)
    offs = torch.tensor([0, n], dtype=torch.int64)
    assert st.host_workspace_bytes("f32", False, n, 1, 4) > st.NOALLOC_STAGING_BYTES
    with pytest.raises(st.SegTopKError) as e:
        st.batched_topk_host_noalloc("f32", keys, offs, 4)
    assert e.value.name == "NOT_SUPPORTED"


def test_calls_allocate_no_device_memory():
    # the property the entry point exists for: after a first call of each
    # shape (which loads the kernels and looks up the staging address), more
    # calls of those shapes leave the device's free memory and torch's
    # allocator untouched
    shapes = [W.random_workload(7100, "f32", [3, 900, 20000], 50, pairs=True, distinct=100, lead=1),
              W.random_workload(7101, "f16", [1, 5000, 70000], 16, "min", pairs=False),
              W.workload1()]

    def call(wl):
        keys, offs, vals, out_k, out_v = host_tensors(wl)
        st.batched_topk_host_noalloc(wl.dtype, keys, offs, wl.k, values=vals, direction=wl.direction,
                                     determinism=wl.determinism, tie_break=wl.tie_break, ordering=wl.ordering,
                                     out_keys=out_k, out_values=out_v, max_segment_len=wl.max_segment_len)

    for wl in shapes:
        call(wl)
    torch.cuda.synchronize()
    free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        for wl in shapes:
            call(wl)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device free memory changed across no-allocation calls"
    assert torch.cuda.memory_allocated() == allocated0
    assert st.read_device_error() == 0
