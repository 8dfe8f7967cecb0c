"""GPU parity of the top-k over one array (segtopk_topk) with the oracle.

The array is one segment for the oracle. The library splits it into up to
304 pieces, keeps each piece's k best and selects the k best of those
("Implement Segmented TopK using Thread-Block-Clusters", section 1.1 names
the non-segmented operation); these cases cover one piece and many, heavy
ties under both tie-breaks, every ordering and determinism mode, int32 and
int64 payloads, and arrays shorter than k.
"""
import numpy as np
import pytest
import torch

import oracle
import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import (NUMPY_SIGNED, ORACLE_THREADS, SENTINEL_BITS, SENTINEL_VALUE, TORCH_VIEW, compare,
                            run_oracle)

pytestmark = pytest.mark.gpu


def run_topk(wl, values=None):
    n, k = wl.num_keys, wl.k
    keys = torch.from_numpy(np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])).cuda()
    kb = W.KEY_BYTES[wl.dtype]
    sent = np.array([SENTINEL_BITS[kb]], dtype=np.uint64).astype({2: np.uint16, 4: np.uint32, 8: np.uint64}[kb])
    out_k = torch.full((k,), int(sent.view(NUMPY_SIGNED[wl.dtype])[0]), dtype=TORCH_VIEW[wl.dtype], device="cuda")
    v = torch.from_numpy(values).cuda() if values is not None else None
    out_v = torch.full((k,), SENTINEL_VALUE, dtype=v.dtype, device="cuda") if v is not None else None
    st.topk(keys, k, values=v, key_dtype=wl.dtype, direction=wl.direction, determinism=wl.determinism,
            tie_break=wl.tie_break, ordering=wl.ordering, out_keys=out_k, out_values=out_v)
    torch.cuda.synchronize()
    assert st.read_device_error() == 0
    gk = out_k.cpu().numpy().view(W.STORAGE[wl.dtype] if wl.dtype != "i32" else np.uint32)
    if wl.dtype == "i32":
        gk = gk.view(np.int32)
    return gk, (out_v.cpu().numpy() if out_v is not None else None)


def array_workload(seed, dtype, n, k, direction, det, tie, ordering, distinct=None, pairs=True):
    wl = W.random_workload(seed, dtype, [n], k, direction, det, tie, ordering, pairs=pairs, distinct=distinct)
    return wl


CASES = [  # dtype, n, k, direction, determinism, tie_break, ordering, distinct
    ("f32", 1000, 8, "max", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted", None),
    ("f32", 5, 64, "min", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted", None),
    ("f16", 50000, 32, "min", "gpu_to_gpu", "prefer_larger_index", "unsorted", 9),
    ("u32", 3_000_000, 1024, "max", "gpu_to_gpu", "prefer_smaller_index", "stable_sorted", 1000),
    ("u32", 3_000_000, 1024, "max", "gpu_to_gpu", "prefer_larger_index", "stable_sorted", 7),
    ("f64", 20_000_000, 256, "max", "gpu_to_gpu", "prefer_smaller_index", "sorted", None),
    ("f32", 20_000_000, 50, "max", "run_to_run", "unspecified", "unsorted", 100000),
    ("bf16", 9_000_000, 300, "min", "not_guaranteed", "unspecified", "stable_sorted", 40),
    ("i32", 7_000_003, 2048, "min", "gpu_to_gpu", "prefer_larger_index", "sorted", 500),
]


@pytest.mark.parametrize("case", CASES, ids=["%s-%d-k%d" % (c[0], c[1], c[2]) for c in CASES])
def test_array_topk_matches_the_oracle(case):
    dtype, n, k, direction, det, tie, ordering, distinct = case
    wl = array_workload(7300 + n % 97 + k, dtype, n, k, direction, det, tie, ordering, distinct=distinct)
    got_k, got_v = run_topk(wl, wl.values)
    want_k, want_v = run_oracle(wl)
    compare(wl, got_k, got_v, want_k, want_v, where="array %s n=%d k=%d" % (dtype, n, k))


def test_array_topk_int64_values():
    wl = array_workload(7400, "f32", 5_000_000, 100, "max", "gpu_to_gpu", "prefer_larger_index",
                        "stable_sorted", distinct=2000, pairs=False)
    vals64 = np.random.Generator(np.random.PCG64(7401)).integers(-2**62, 2**62, size=wl.num_keys, dtype=np.int64)
    got_k, got_v = run_topk(wl, vals64)
    pos_wl = W.Workload(wl.name, wl.dtype, wl.keys, np.arange(wl.num_keys, dtype=np.int32), wl.offsets, wl.k,
                        wl.direction, wl.determinism, wl.tie_break, wl.ordering)
    want_k, pos = run_oracle(pos_wl)
    assert np.array_equal(got_k, want_k)
    assert np.array_equal(got_v, vals64[pos])


def test_array_topk_2_27_keys():
    # the oracle on the subset of keys at least the k-th best (in array order,
    # original positions as values): every other key has k better keys
    n, k = (1 << 27) + 3, 1000
    keys = np.random.Generator(np.random.PCG64(7500)).integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # about 500 keys lie above V and 1342 keys equal V: the k-th key is a tie
    keys[::100000] = np.uint32(2**32 - 16000)
    wl = W.Workload("u32 2^27+3", "u32", keys, None, np.array([0, n], dtype=np.int64), k, "max", "gpu_to_gpu",
                    "prefer_larger_index", "stable_sorted")
    pos = np.arange(n, dtype=np.int32)
    got_k, got_v = run_topk(wl, pos)
    kth = np.partition(keys, n - k)[n - k]
    sub = np.nonzero(keys >= kth)[0]
    want_k, want_v = oracle.batched_topk("u32", keys[sub], sub.astype(np.int32),
                                         np.array([0, sub.size], dtype=np.int64), k, "max", "prefer_larger_index",
                                         threads=ORACLE_THREADS)
    assert np.array_equal(got_k, want_k)
    assert np.array_equal(got_v, want_v)
