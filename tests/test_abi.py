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
    assert call(lib, keys=18) == 4               # misaligned keys
    assert call(lib, k=B.MAX_K + 1) == 3
    assert call(lib, max_len=(1 << 31)) == 3


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
    a = st.host_workspace_bytes("f32", False, 1000, 10, 8)
    b = st.host_workspace_bytes("f32", True, 1000, 10, 8)
    assert a >= 4000 + 88 + 320 and b >= a + 4000 + 320
    assert st.host_workspace_bytes("f32", True, -1, 10, 8) == 0


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
