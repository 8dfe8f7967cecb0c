"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the CPU oracle on the same seeded arrays, then compare."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import segmented_radix_top_gb300 as st
from segmented_radix_top_gb300 import workloads as W

TORCH_VIEW = {"f16": torch.int16, "bf16": torch.int16, "f32": torch.int32, "f64": torch.int64,
              "u32": torch.int32, "i32": torch.int32}
NUMPY_SIGNED = {"f16": np.int16, "bf16": np.int16, "f32": np.int32, "f64": np.int64,
                "u32": np.int32, "i32": np.int32}
SENTINEL_BITS = {2: 0x5A5A, 4: 0x5A5A5A5A, 8: 0x5A5A5A5A5A5A5A5A}
SENTINEL_VALUE = -123456789
ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))


def to_device_keys(wl: W.Workload, device="cuda") -> torch.Tensor:
    arr = np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])
    return torch.from_numpy(arr).to(device)


def run_gpu(wl: W.Workload, cluster_width: int = 0, max_segment_len="auto", device="cuda",
            values: np.ndarray | None = "workload", keys_t=None, stream=None, small_segment_max_len: int = 0,
            team_segment_max_len: int = 0, lib=None):
    """Returns (out_key_bits [S*k] storage dtype, out_values or None) as numpy."""
    if keys_t is None:
        keys_t = to_device_keys(wl, device)
    offs = torch.from_numpy(wl.offsets).to(device)
    vals = wl.values if (isinstance(values, str) and values == "workload") else values
    vals_t = torch.from_numpy(vals).to(device) if vals is not None else None
    S, k = wl.num_segments, wl.k
    kb = W.KEY_BYTES[wl.dtype]
    sent = np.array([SENTINEL_BITS[kb]], dtype=W.STORAGE[wl.dtype] if wl.dtype != "i32" else np.uint32)
    sent_signed = int(sent.view(NUMPY_SIGNED[wl.dtype])[0])
    out_k = torch.full((max(S, 0) * k,), sent_signed, dtype=TORCH_VIEW[wl.dtype], device=device)
    out_v = torch.full((max(S, 0) * k,), SENTINEL_VALUE, dtype=torch.int32, device=device) \
        if vals_t is not None else None
    ml = wl.max_segment_len if max_segment_len == "auto" else max_segment_len
    st.batched_topk(keys_t, offs, k, values=vals_t, key_dtype=wl.dtype, direction=wl.direction,
                    determinism=wl.determinism, tie_break=wl.tie_break, ordering=wl.ordering,
                    out_keys=out_k, out_values=out_v, max_segment_len=ml,
                    cluster_width=cluster_width, stream=stream, small_segment_max_len=small_segment_max_len,
                    team_segment_max_len=team_segment_max_len, lib=lib)
    torch.cuda.synchronize()
    gk = out_k.cpu().numpy().view(W.STORAGE[wl.dtype] if wl.dtype != "i32" else np.uint32)
    if wl.dtype == "i32":
        gk = gk.view(np.int32)
    gv = out_v.cpu().numpy() if out_v is not None else None
    return gk, gv


def run_oracle(wl: W.Workload, values: np.ndarray | None = "workload"):
    vals = wl.values if (isinstance(values, str) and values == "workload") else values
    kb = W.KEY_BYTES[wl.dtype]
    st_dtype = W.STORAGE[wl.dtype]
    sent = np.array([SENTINEL_BITS[kb]], dtype=st_dtype if wl.dtype != "i32" else np.uint32)
    if wl.dtype == "i32":
        sent = sent.view(np.int32)
    out_k = np.full(wl.num_segments * wl.k, sent[0], dtype=st_dtype)
    out_v = np.full(wl.num_segments * wl.k, SENTINEL_VALUE, dtype=np.int32) if vals is not None else None
    return oracle.batched_topk(wl.dtype, wl.keys, vals, wl.offsets, wl.k, wl.direction, wl.tie_break,
                               out_keys=out_k, out_values=out_v, threads=ORACLE_THREADS)


SIGN_BIT = {2: 0x8000, 4: 0x80000000, 8: 1 << 63}
FLOAT_TYPES = ("f16", "bf16", "f32", "f64")


def canonical(wl: W.Workload, bits: np.ndarray) -> np.ndarray:
    """Key bits with -0.0 replaced by +0.0 (equal keys compare equal), as int64
    (uint64 for 64-bit keys)."""
    b = bits.astype(np.uint64 if bits.dtype == np.uint64 else np.int64)
    if wl.dtype in FLOAT_TYPES:
        kb = W.KEY_BYTES[wl.dtype]
        neg0 = np.uint64(SIGN_BIT[kb]) if b.dtype == np.uint64 else np.int64(SIGN_BIT[kb])
        b = np.where(b == neg0, b.dtype.type(0), b)
    return b


def compare(wl: W.Workload, got_k, got_v, want_k, want_v, where=""):
    """Parity with the oracle, by the contract of each mode ("Top-K:
    Determinism, Tie-Breaking, and Output Ordering").

    Slots past min(k, n) must still hold the caller's fill (the oracle leaves
    them untouched too).
    gpu_to_gpu / run_to_run (the set is fixed):
      stable_sorted: every slot equal (key bits and values);
      sorted: keys in the same order up to equal keys (+0.0 and -0.0 count
        as equal), and the per-segment multiset of (key bits, value) equal;
      unsorted: the per-segment multiset of (key bits, value) equal.
    not_guaranteed (any valid subset of boundary ties): the per-segment
      multiset of keys (+0.0 = -0.0) equal, keys in order when sorted, and
      every (key bits, value) output a distinct element of its segment.
    """
    S, k = wl.num_segments, wl.k
    if S == 0 or k == 0:
        return
    gk = got_k.reshape(S, k)
    wk = want_k.reshape(S, k)
    gv = got_v.reshape(S, k) if got_v is not None else None
    wv = want_v.reshape(S, k) if want_v is not None else None
    m = np.minimum(wl.lengths, k)
    slot = np.arange(k)[None, :]
    live = slot < m[:, None]
    # untouched tail slots
    bad = np.nonzero(~live & (gk != wk))
    assert bad[0].size == 0, "%s: tail slot overwritten in segment %d" % (where, bad[0][0])
    if gv is not None:
        bad = np.nonzero(~live & (gv != wv))
        assert bad[0].size == 0, "%s: tail value overwritten in segment %d" % (where, bad[0][0])
    if wl.ordering == "stable_sorted" and wl.determinism != "not_guaranteed":
        bad = np.nonzero(live & (gk != wk))
        assert bad[0].size == 0, "%s: key mismatch seg %d slot %d: got %x want %x" % (
            where, bad[0][0], bad[1][0], int(gk[bad][0]), int(wk[bad][0]))
        if gv is not None:
            bad = np.nonzero(live & (gv != wv))
            assert bad[0].size == 0, "%s: value mismatch seg %d slot %d: got %d want %d" % (
                where, bad[0][0], bad[1][0], int(gv[bad][0]), int(wv[bad][0]))
        return
    seg = np.repeat(np.arange(S), k).reshape(S, k)
    g_can, w_can = canonical(wl, gk), canonical(wl, wk)
    if wl.ordering != "unsorted":
        bad = np.nonzero(live & (g_can != w_can))
        assert bad[0].size == 0, "%s: keys out of order, seg %d slot %d" % (where, bad[0][0], bad[1][0])
    g_bits = gk[live].astype(np.int64) if gk.dtype != np.uint64 else gk[live]
    w_bits = wk[live].astype(np.int64) if wk.dtype != np.uint64 else wk[live]
    g_seg = seg[live]
    if wl.determinism == "not_guaranteed":
        go = np.lexsort((g_can[live], g_seg))
        wo = np.lexsort((w_can[live], g_seg))
        assert np.array_equal(g_can[live][go], w_can[live][wo]), "%s: key multiset differs" % where
        check_real_elements(wl, gk, gv, live, where)
        return
    if gv is not None:
        go = np.lexsort((gv[live], g_bits, g_seg))
        wo = np.lexsort((wv[live], w_bits, g_seg))
        assert np.array_equal(gv[live][go], wv[live][wo]), "%s: value multiset differs" % where
    else:
        go = np.lexsort((g_bits, g_seg))
        wo = np.lexsort((w_bits, g_seg))
    assert np.array_equal(g_bits[go], w_bits[wo]), "%s: key multiset differs" % where


def check_real_elements(wl: W.Workload, gk, gv, live, where):
    """Every output (key bits, value) of a segment is an element of that
    segment, each element used at most once."""
    from collections import Counter
    for s in range(wl.num_segments):
        n = int(live[s].sum())
        if n == 0:
            continue
        b, e = int(wl.offsets[s]), int(wl.offsets[s + 1])
        keys = wl.keys[b:e]
        vals = wl.values[b:e] if (wl.values is not None and gv is not None) else np.zeros(e - b, dtype=np.int64)
        have = Counter(zip(keys.tolist(), vals.tolist()))
        outv = gv[s, :n].tolist() if (wl.values is not None and gv is not None) else [0] * n
        used = Counter(zip(gk[s, :n].astype(keys.dtype).tolist(), outv))
        for item, c in used.items():
            assert have.get(item, 0) >= c, "%s: seg %d output %r is not an element (or repeats)" % (
                where, s, item)


def check_workload(wl: W.Workload, cluster_width: int = 0, where: str = "", **kw):
    got_k, got_v = run_gpu(wl, cluster_width=cluster_width, **kw)
    want_k, want_v = run_oracle(wl, values=kw.get("values", "workload"))
    compare(wl, got_k, got_v, want_k, want_v, where=where or wl.name)
    err = st.read_device_error(lib=kw.get("lib"))
    assert err == 0, "device error word %#x" % err
    return got_k, got_v
