"""Host-only checks of the C ABI: the library loads, exports every function
include/segtopk.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import _binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "segtopk.h")


@pytest.fixture(scope="module")
def lib():
    st.build()
    return st.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(segtopk_\w+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "segtopk_batched_topk" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), "missing export %s" % n


def call(lib, dtype=2, keys=16, values=None, offs=64, nseg=1, k=4, direction=0, det=2, tie=1,
         ordering=2, out_keys=128, out_values=None, max_len=100):
    vp = ctypes.c_void_p
    return lib.segtopk_batched_topk(dtype, vp(keys) if keys else None, vp(values) if values else None,
                                    vp(offs) if offs else None, nseg, k, direction, det, tie, ordering,
                                    vp(out_keys) if out_keys else None,
                                    vp(out_values) if out_values else None, max_len, None)


def test_invalid_enums(lib):
    assert call(lib, dtype=9) == 1
    assert call(lib, direction=2) == 1
    assert call(lib, det=3) == 1
    assert call(lib, tie=3) == 1
    assert call(lib, ordering=5) == 1


def test_invalid_combinations(lib):
    # a concrete tie-break needs gpu_to_gpu
    assert call(lib, det=0, tie=1) == 2
    assert call(lib, det=1, tie=2) == 2
    assert call(lib, det=0, tie=2) == 2


def test_noop_and_sizes(lib):
    assert call(lib, nseg=0) == 0
    assert call(lib, k=0) == 0
    assert call(lib, nseg=-1) == 1
    assert call(lib, k=-3) == 1
    assert call(lib, keys=0) == 1
    assert call(lib, offs=0) == 1
    assert call(lib, out_keys=0) == 1
    assert call(lib, values=256) == 1            # values without out_values
    assert call(lib, out_values=256) == 1        # out_values without values
    assert call(lib, keys=18) == 4               # keys not aligned to the element size (f32)
    assert call(lib, dtype=0, keys=17) == 4      # f16 keys at an odd address
    assert call(lib, dtype=3, keys=20) == 4      # f64 keys 4-byte aligned only
    assert call(lib, k=B.MAX_K + 1) == 3
    assert call(lib, max_len=(1 << 31)) == 3


def test_element_aligned_keys_pass_validation(lib):
    # keys need only element alignment: an offset view of a larger array is
    # accepted (without a device the call then fails at the device query)
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake pointers must not reach a launch on a machine with a GPU")
    assert call(lib, keys=20) == 5               # f32 at 4-byte alignment: validated, then no device
    assert call(lib, dtype=0, keys=18) == 5      # f16 at 2-byte alignment


def test_diagnostics_are_off_in_the_ordinary_build(lib):
    arr = (ctypes.c_uint64 * 16)()
    assert lib.segtopk_read_stats(arr, 16) == 3
    assert lib.segtopk_set_test_hooks(1000, 16) == 3
    one = (ctypes.c_int * 1)(0)
    assert lib.segtopk_test_device_prep(1, one, (ctypes.c_uint32 * 1)(1024), one, (ctypes.c_uint32 * 1)()) == 3


def test_launch_preparation_is_kept_per_device():
    # function attributes belong to each device's copy of a kernel: a second
    # GPU in the same process needs its own opt-in, wide-cluster permission
    # and carveout, however far the first one was raised
    seq = [(0, 50000, 1),    # raise device 0's opt-in
           (1, 50000, 1),    # device 1 needs its own
           (0, 40000, 2),    # already granted on device 0
           (0, 90000, 16),   # a larger opt-in and clusters wider than 8
           (1, 90000, 16),   # both again on device 1
           (1, 90000, 16),   # nothing left to do
           (1, 60000, 12),   # smaller, and wide clusters already allowed
           (0, 0, 0),        # warp kernel on device 0: carveout once
           (0, 0, 0),
           (3, 0, -1),       # and on device 3
           (64, 1024, 1),    # ordinals outside 0..63 are refused
           (-1, 1024, 1)]
    got = B.test_device_prep(seq)
    assert got == [1, 1, 0, 3, 3, 0, 0, 4, 0, 4, 0xFFFFFFFF, 0xFFFFFFFF]
    assert B.test_device_prep([]) == []


def test_status_strings(lib):
    for code in range(7):
        assert lib.segtopk_status_string(code)
    assert lib.segtopk_status_string(99) == b"unknown status"


def test_options_validation(lib):
    o = B.Options()
    o.cluster_width = 17
    vp = ctypes.c_void_p
    rc = lib.segtopk_batched_topk_ex(2, vp(16), None, vp(64), 1, 4, 0, 2, 1, 2, vp(128), None, 100,
                                     ctypes.byref(o), None)
    assert rc == 1
    o.cluster_width = 0
    o.reserved[3] = 1
    rc = lib.segtopk_batched_topk_ex(2, vp(16), None, vp(64), 1, 4, 0, 2, 1, 2, vp(128), None, 100,
                                     ctypes.byref(o), None)
    assert rc == 1


def test_workspace_bytes(lib):
    # keys, offsets and output keys; pairs add the selected source indices
    # (values stay on the host)
    a = st.host_workspace_bytes("f32", False, 1000, 10, 8)
    b = st.host_workspace_bytes("f32", True, 1000, 10, 8)
    assert a >= 4000 + 88 + 320 and b >= a + 320
    assert b < a + 4000  # no device copy of the values
    assert st.host_workspace_bytes("f32", True, -1, 10, 8) == 0
    assert st.host_workspace_bytes("f64", False, 1 << 62, 1, 8) == 0  # byte count would overflow


def _host_call(lib, offsets, values=False, noalloc=False, k=4):
    """Host-buffer entry points with real host arrays and a fake (never
    touched) device workspace: the checks below fail before any copy."""
    import numpy as np
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    n = max(int(offs.max()), 1)
    keys = np.zeros(n, dtype=np.float32)
    vals = np.zeros(n, dtype=np.int32) if values else None
    nseg = len(offs) - 1
    ok = np.zeros(nseg * k, dtype=np.float32)
    ov = np.zeros(nseg * k, dtype=np.int32) if values else None
    vp = ctypes.c_void_p
    args = [2, vp(keys.ctypes.data), vp(vals.ctypes.data) if values else None, vp(offs.ctypes.data), nseg, k,
            0, 2, 1, 2, vp(ok.ctypes.data), vp(ov.ctypes.data) if values else None, -1]
    if noalloc:
        return lib.segtopk_batched_topk_host_noalloc(*args, None)
    return lib.segtopk_batched_topk_host(*args, vp(256), 1 << 30, None)


def test_host_path_rejects_negative_offsets(lib):
    # a negative offset would make the kernel read before the key array
    for noalloc in (False, True):
        for offs in ([-4, 10], [0, 5, -1, 8], [-1, -1]):
            for values in (False, True):
                assert _host_call(lib, offs, values=values, noalloc=noalloc) == 1
                assert lib.segtopk_last_launch_count() == 0


def test_host_path_rejects_unaligned_workspace(lib):
    import numpy as np
    keys = np.zeros(8, dtype=np.float32)
    offs = np.array([0, 8], dtype=np.int64)
    ok = np.zeros(4, dtype=np.float32)
    vp = ctypes.c_void_p
    rc = lib.segtopk_batched_topk_host(2, vp(keys.ctypes.data), None, vp(offs.ctypes.data), 1, 4, 0, 2, 1, 2,
                                       vp(ok.ctypes.data), None, -1, vp(256 + 16), 1 << 20, None)
    assert rc == 4


def _header_text():
    return re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)


def _header_define(name):
    m = re.search(r"#define\s+%s\s+\(?([0-9u\s*]+)\)?" % name, _header_text())
    assert m, name
    return eval(m.group(1).replace("u", ""))  # plain integer products only


def test_options_struct_matches_header():
    body = re.search(r"typedef struct \{(.*?)\} segtopk_options;", _header_text(), flags=re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+)(?:\[(\d+)\])?;", body)
    want = [(name, ctypes.c_int32 * int(n) if n else ctypes.c_int32) for name, n in fields]
    got = B.Options._fields_
    assert [n for n, _ in got] == [n for n, _ in want]
    assert ctypes.sizeof(B.Options) == sum(ctypes.sizeof(t) for _, t in want) == 32


def test_duplicated_constants_match_header():
    import bench
    assert B.MAX_K == _header_define("SEGTOPK_MAX_K")
    assert B.NOALLOC_STAGING_BYTES == _header_define("SEGTOPK_NOALLOC_STAGING_BYTES")
    assert bench.SMALL_SEGMENT_DEFAULT == _header_define("SEGTOPK_SMALL_SEGMENT_DEFAULT")
    assert bench.TEAM_SEGMENT_FEW == _header_define("SEGTOPK_TEAM_SEGMENT_FEW")


def test_options_reject_nonzero_reserved_fields(lib):
    vp = ctypes.c_void_p
    for i in range(len(B.Options().reserved)):
        o = B.Options()
        o.reserved[i] = 7
        rc = lib.segtopk_batched_topk_ex(2, vp(16), None, vp(64), 1, 4, 0, 2, 1, 2, vp(128), None, 100,
                                         ctypes.byref(o), None)
        assert rc == 1
