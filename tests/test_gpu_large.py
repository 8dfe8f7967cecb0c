"""GPU parity for 64-bit payloads and long segments.

"Implement Segmented TopK using Thread-Block-Clusters", section 10 "Known
limitations and future work", names wider value types and segments beyond
its 2^21-key cap. Here:

* int64 values (segtopk_batched_topk_values) on every path -- single warp,
  team of warps, CTA, cluster -- compared with the oracle, which is run with
  each element's position as its value: the expected 64-bit value of a slot
  is the payload at the position the oracle selected;
* one segment of 3 * 2^21 + 17 keys at an unaligned start, every slot
  compared with the oracle, at automatic and forced cluster widths;
* one segment of 2^28 + 5 keys. The oracle runs on the subset of keys at
  least as good as the k-th best (found by a partition on the host), in
  their original order and with their original positions as values: every
  key outside the subset has k better keys, and the subset keeps the order
  that decides ties, so its top-k is the segment's.
"""
import numpy as np
import pytest
import torch

import oracle
import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W
from tests.gpu_util import (NUMPY_SIGNED, ORACLE_THREADS, SENTINEL_BITS, SENTINEL_VALUE, TORCH_VIEW, compare,
                            run_gpu, run_oracle)

pytestmark = pytest.mark.gpu


def with_positions(wl):
    """The workload with int32 values = element position (for the oracle)."""
    return W.Workload(wl.name, wl.dtype, wl.keys, np.arange(wl.num_keys, dtype=np.int32), wl.offsets, wl.k,
                      wl.direction, wl.determinism, wl.tie_break, wl.ordering)


def run_gpu64(wl, vals64, **kw):
    keys = torch.from_numpy(np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])).cuda()
    offs = torch.from_numpy(wl.offsets).cuda()
    v = torch.from_numpy(vals64).cuda()
    S, k = wl.num_segments, wl.k
    kb = W.KEY_BYTES[wl.dtype]
    sent = np.array([SENTINEL_BITS[kb]], dtype=np.uint64).astype({2: np.uint16, 4: np.uint32, 8: np.uint64}[kb])
    out_k = torch.full((S * k,), int(sent.view(NUMPY_SIGNED[wl.dtype])[0]), dtype=TORCH_VIEW[wl.dtype],
                       device="cuda")
    out_v = torch.full((S * k,), SENTINEL_VALUE, dtype=torch.int64, device="cuda")
    st.batched_topk(keys, offs, k, values=v, key_dtype=wl.dtype, direction=wl.direction,
                    determinism=wl.determinism, tie_break=wl.tie_break, ordering=wl.ordering, out_keys=out_k,
                    out_values=out_v, max_segment_len=wl.max_segment_len, **kw)
    torch.cuda.synchronize()
    assert st.read_device_error() == 0
    gk = out_k.cpu().numpy().view(W.STORAGE[wl.dtype] if wl.dtype != "i32" else np.uint32)
    if wl.dtype == "i32":
        gk = gk.view(np.int32)
    return gk, out_v.cpu().numpy()


def expected64(wl, vals64):
    want_k, pos = run_oracle(with_positions(wl))
    live = np.arange(wl.k)[None, :] < np.minimum(wl.lengths, wl.k)[:, None]
    want_v = np.full(pos.shape, SENTINEL_VALUE, dtype=np.int64)
    want_v[live.reshape(-1)] = vals64[pos[live.reshape(-1)]]
    return want_k, want_v


PATHS = [  # (k, cluster_width, small_segment_max_len, team_segment_max_len)
    (8, 0, 100000, -1), (16, 0, -1, 100000), (50, 1, -1, -1), (300, 3, -1, -1), (1024, 0, 0, 0)]


@pytest.mark.parametrize("dtype", ["f32", "f64", "f16", "u32"])
@pytest.mark.parametrize("path", PATHS, ids=["warp", "team", "cta", "cluster", "auto"])
def test_int64_values(dtype, path):
    k, width, small, team = path
    g = np.random.Generator(np.random.PCG64(77))
    lengths = [0, 3, 9, 100, 2000, 9001, 40000, 131075]
    for i, (tie, ordering) in enumerate([("prefer_smaller_index", "stable_sorted"),
                                         ("prefer_larger_index", "unsorted")]):
        wl = W.random_workload(6000 + i, dtype, lengths, k, "max" if i else "min", "gpu_to_gpu", tie, ordering,
                               pairs=False, distinct=300, lead=i + 1)
        vals64 = g.integers(-2**62, 2**62, size=wl.num_keys, dtype=np.int64)
        got_k, got_v = run_gpu64(wl, vals64, cluster_width=width, small_segment_max_len=small,
                                 team_segment_max_len=team)
        want_k, want_v = expected64(wl, vals64)
        compare(wl, got_k, got_v, want_k, want_v, where="int64 %s k=%d %s" % (dtype, k, ordering))


@pytest.mark.parametrize("width", [0, 1, 16])
def test_segment_beyond_2_21_keys(width):
    n = 3 * (1 << 21) + 17
    for i, (dtype, k, tie, ordering, direction) in enumerate([
            ("f32", 100, "prefer_smaller_index", "stable_sorted", "max"),
            ("u32", 1024, "prefer_larger_index", "unsorted", "min")]):
        wl = W.random_workload(6100 + i, dtype, [5, n, 70000], k, direction, "gpu_to_gpu", tie, ordering,
                               pairs=True, distinct=1 << 16, lead=3)
        got_k, got_v = run_gpu(wl, cluster_width=width)
        want_k, want_v = run_oracle(wl)
        compare(wl, got_k, got_v, want_k, want_v, where="n=3*2^21+17 %s C=%d" % (dtype, width))


def test_segment_of_2_28_keys():
    n = (1 << 28) + 5
    k = 64
    g = np.random.Generator(np.random.PCG64(6200))
    keys = g.integers(0, 2**32, size=n + 1, dtype=np.uint64).astype(np.uint32)
    offs = np.array([1, n + 1], dtype=np.int64)  # starts one element in: unaligned
    wl = W.Workload("u32 2^28+5", "u32", keys, None, offs, k, "max", "gpu_to_gpu", "prefer_smaller_index",
                    "stable_sorted")
    pos_t = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    got_k, got_v = run_gpu(wl, values=None, max_segment_len=n)
    keys_t = torch.from_numpy(keys.view(np.int32)).cuda()
    out_k = torch.empty(k, dtype=torch.int32, device="cuda")
    out_v = torch.empty(k, dtype=torch.int32, device="cuda")
    st.batched_topk(keys_t, torch.from_numpy(offs).cuda(), k, values=pos_t, key_dtype="u32", direction="max",
                    determinism="gpu_to_gpu", tie_break="prefer_smaller_index", ordering="stable_sorted",
                    out_keys=out_k, out_values=out_v, max_segment_len=n)
    torch.cuda.synchronize()
    assert st.read_device_error() == 0
    assert np.array_equal(out_k.cpu().numpy().view(np.uint32), got_k[:k])
    # the subset of keys at least the k-th largest, in original order
    seg = keys[1:]
    kth = np.partition(seg, n - k)[n - k]
    sub_pos = np.nonzero(seg >= kth)[0]
    assert sub_pos.size >= k
    sub = W.Workload("subset", "u32", seg[sub_pos], (sub_pos + 1).astype(np.int32),
                     np.array([0, sub_pos.size], dtype=np.int64), k, "max", "gpu_to_gpu", "prefer_smaller_index",
                     "stable_sorted")
    want_k, want_pos = oracle.batched_topk("u32", sub.keys, sub.values, sub.offsets, k, "max",
                                           "prefer_smaller_index", threads=ORACLE_THREADS)
    assert np.array_equal(got_k[:k], want_k), "keys differ from the oracle's"
    assert np.array_equal(out_v.cpu().numpy(), want_pos), "positions differ from the oracle's"
