"""Pins that tie the CPU oracle to facts fixed outside itself.

Each check is independent of the oracle's C code:
  * the worked example printed on "Top-K: Determinism, Tie-Breaking, and Output
    Ordering" (golden fixture);
  * brute force over the closed-form rank definition of top-k on tiny inputs
    (pure Python, numbers decoded by numpy / torch, not by the oracle);
  * a library special case: numpy's lexsort over the decoded numbers;
  * exhaustive decoding of every 16-bit float pattern against numpy / torch;
  * the invariants the contract states (count, dominance, -0.0 survival).
A plausible slip in the oracle (a flipped direction, a swapped tie rule, a
dropped index tie-break, +/-0 treated as different, a wrong output order or
an off-by-one in m) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from segmented_radix_top_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DTYPES = ["f16", "bf16", "f32", "f64", "u32", "i32"]
TIES = ["unspecified", "prefer_smaller_index", "prefer_larger_index"]


def decode(dtype, bits):
    """Numbers from raw bits via numpy/torch (independent of the oracle)."""
    bits = np.asarray(bits)
    if dtype == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if dtype == "bf16":
        t = torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)
        return t.to(torch.float64).numpy()
    if dtype == "f32":
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "f64":
        return bits.astype(np.uint64).view(np.float64)
    if dtype == "u32":
        return bits.astype(np.uint32).astype(np.float64)
    return bits.astype(np.int32).astype(np.float64)


def brute_force(vals, k, direction, tie):
    """Top-k by the rank definition: element i is selected iff
    #{j better than i} + #{j equal to i and preferred over i} < k; its stable
    output position is #{selected j better than i, or equal with j < i}."""
    n = len(vals)
    larger_wins = tie == "prefer_larger_index"

    def better(a, b):
        return vals[a] > vals[b] if direction == "max" else vals[a] < vals[b]

    rank = []
    for i in range(n):
        r = 0
        for j in range(n):
            if j == i:
                continue
            if better(j, i) or (vals[j] == vals[i] and ((j > i) if larger_wins else (j < i))):
                r += 1
        rank.append(r)
    sel = [i for i in range(n) if rank[i] < k]
    pos = {}
    for i in sel:
        pos[i] = sum(1 for j in sel if j != i and (better(j, i) or (vals[j] == vals[i] and j < i)))
    assert sorted(pos.values()) == list(range(len(sel)))
    return sorted(sel, key=lambda i: pos[i])


def run_oracle(wl, threads=1):
    return oracle.batched_topk(wl.dtype, wl.keys, wl.values, wl.offsets, wl.k, wl.direction,
                               wl.tie_break, threads=threads)


# ---------------------------------------------------------------- worked example

def load_worked_example():
    spec = {"results": []}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "keys":
                spec["keys"] = [int(x) for x in parts[1:]]
            elif parts[0] == "k":
                spec["k"] = int(parts[1])
            elif parts[0] == "direction":
                spec["direction"] = parts[1]
            elif parts[0] == "result":
                items = [tuple(int(v) for v in it.split("@")) for it in parts[3:]]
                spec["results"].append((parts[1], parts[2], items))
    return spec


@pytest.mark.parametrize("dtype", DTYPES)
def test_worked_example(dtype):
    spec = load_worked_example()
    assert len(spec["results"]) == 4
    keys = np.array(spec["keys"], dtype=np.float64)
    if dtype == "f16":
        bits = W.f16_bits(keys)
    elif dtype == "bf16":
        bits = W.bf16_bits(keys.astype(np.float32))
    elif dtype == "f32":
        bits = W.f32_bits(keys)
    elif dtype == "f64":
        bits = W.f64_bits(keys)
    elif dtype == "u32":
        bits = keys.astype(np.uint32)
    else:
        bits = keys.astype(np.int32)
    vals = np.arange(len(keys), dtype=np.int32)  # value = source index
    offs = np.array([0, len(keys)], dtype=np.int64)
    for tie, order, items in spec["results"]:
        ok, ov = oracle.batched_topk(dtype, bits, vals, offs, spec["k"], spec["direction"], tie)
        got = [(int(round(float(decode(dtype, [b])[0]))), int(v)) for b, v in zip(ok, ov)]
        if order == "set":
            assert sorted(got, key=lambda t: t[1]) == sorted(items, key=lambda t: t[1])
        else:
            assert got == items


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("direction", ["max", "min"])
@pytest.mark.parametrize("tie", TIES)
def test_brute_force_rank_definition(dtype, direction, tie):
    g = np.random.Generator(np.random.PCG64(77))
    for trial in range(12):
        lengths = g.integers(0, 24, size=4)
        k = int(g.integers(0, 26))
        distinct = [None, 3, 6][trial % 3]
        wl = W.random_workload(int(g.integers(1 << 30)), dtype, lengths, k, direction,
                               tie_break=tie, distinct=distinct, lead=int(g.integers(0, 5)))
        ok, ov = run_oracle(wl)
        nums = decode(dtype, wl.keys)
        for s in range(wl.num_segments):
            b, e = int(wl.offsets[s]), int(wl.offsets[s + 1])
            want = brute_force(list(nums[b:e]), k, direction, tie)
            m = len(want)
            assert m == min(k, e - b)
            got_bits = ok[s * k: s * k + m]
            got_vals = ov[s * k: s * k + m]
            assert list(got_bits) == [wl.keys[b + i] for i in want]
            assert list(got_vals) == [wl.values[b + i] for i in want]


def test_brute_force_signed_zero_ties():
    """Only +0.0 / -0.0 and a few other keys: the zeros tie, bits survive."""
    g = np.random.Generator(np.random.PCG64(5))
    for dtype, direction, tie in itertools.product(["f16", "bf16", "f32", "f64"], ["max", "min"], TIES):
        x = g.choice(np.array([0.0, -0.0, 1.0, -1.0]), size=30)
        x[g.random(30) < 0.5] = g.choice([0.0, -0.0])
        bits = {"f16": W.f16_bits, "f32": W.f32_bits, "f64": W.f64_bits,
                "bf16": lambda v: W.bf16_bits(v.astype(np.float32))}[dtype](x)
        vals = np.arange(30, dtype=np.int32)
        for k in (1, 5, 13, 29):
            ok, ov = oracle.batched_topk(dtype, bits, vals, np.array([0, 30]), k, direction, tie)
            want = brute_force(list(decode(dtype, bits)), k, direction, tie)
            assert list(ov) == want
            assert list(ok) == [bits[i] for i in want]  # -0.0 bit patterns survive


# ---------------------------------------------------------------- library special case

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("direction", ["max", "min"])
@pytest.mark.parametrize("tie", ["prefer_smaller_index", "prefer_larger_index"])
def test_numpy_lexsort(dtype, direction, tie):
    g = np.random.Generator(np.random.PCG64(11))
    lengths = g.integers(0, 3000, size=12)
    wl = W.random_workload(3, dtype, lengths, 97, direction, tie_break=tie,
                           distinct=40 if dtype != "f64" else None, lead=3)
    ok, ov = run_oracle(wl, threads=4)
    nums = decode(dtype, wl.keys)
    sign = -1.0 if direction == "max" else 1.0
    for s in range(wl.num_segments):
        b, e = int(wl.offsets[s]), int(wl.offsets[s + 1])
        v = nums[b:e] * sign
        idx = np.arange(e - b)
        sec = -idx if tie == "prefer_larger_index" else idx
        sel = np.lexsort((sec, v))[: min(97, e - b)]
        out = sel[np.lexsort((sel, v[sel]))]
        m = len(out)
        assert np.array_equal(ok[s * 97: s * 97 + m], wl.keys[b + out])
        assert np.array_equal(ov[s * 97: s * 97 + m], wl.values[b + out])


# ---------------------------------------------------------------- decoding

def test_decode_f16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32)
    want = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.decode_f16(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_exhaustive():
    bits = np.arange(65536, dtype=np.uint32)
    want = decode("bf16", bits.astype(np.uint16))
    got = np.array([oracle.decode_bf16(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ---------------------------------------------------------------- NaN reading

def test_nan_reading():
    """NaN order is a reading (the pages are silent): +NaN above +inf, -NaN
    below -inf; same-sign NaNs order by payload (descending for -NaN)."""
    pos_nan_small = 0x7FC00001
    pos_nan_big = 0x7FC00100
    neg_nan_small = 0xFFC00001
    neg_nan_big = 0xFFC00100
    inf, ninf = 0x7F800000, 0xFF800000
    bits = np.array([inf, pos_nan_small, ninf, neg_nan_big, pos_nan_big, neg_nan_small, 0],
                    dtype=np.uint32)
    vals = np.arange(7, dtype=np.int32)
    offs = np.array([0, 7])
    _, ov = oracle.batched_topk("f32", bits, vals, offs, 7, "max", "prefer_smaller_index")
    assert list(ov) == [4, 1, 0, 6, 2, 5, 3]
    _, ov = oracle.batched_topk("f32", bits, vals, offs, 7, "min", "prefer_smaller_index")
    assert list(ov) == [3, 5, 2, 6, 0, 1, 4]


# ---------------------------------------------------------------- contract invariants

@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_invariants_on_workload_shapes(cfg):
    shrink = {1: {}, 2: dict(segments=4, seg_len=20000), 3: dict(segments=200, max_len=6000),
              4: dict(segments=2, seg_len=65536), 5: dict(segments=8, seg_len=4096)}[cfg]
    wl = W.by_number(cfg, **shrink)
    vals = np.arange(wl.num_keys, dtype=np.int32)  # values = global position, to locate picks
    k = wl.k
    ok, ov = oracle.batched_topk(wl.dtype, wl.keys, vals, wl.offsets, k, wl.direction,
                                 wl.tie_break, threads=4)
    nums = decode(wl.dtype, wl.keys)
    for s in range(wl.num_segments):
        b, e = int(wl.offsets[s]), int(wl.offsets[s + 1])
        m = min(k, e - b)
        picks = ov[s * k: s * k + m]
        assert len(set(picks.tolist())) == m and np.all((picks >= b) & (picks < e))
        assert np.array_equal(ok[s * k: s * k + m], wl.keys[picks])  # bits, incl. -0.0
        chosen = nums[picks]
        rest = np.setdiff1d(np.arange(b, e), picks)
        if len(rest):
            if wl.direction == "max":
                assert chosen.min() >= nums[rest].max()
            else:
                assert chosen.max() <= nums[rest].min()
        # stable-sorted output: keys ordered better-first, equal keys by index
        seq = list(zip(chosen.tolist(), picks.tolist()))
        for (a, ia), (c, ic) in zip(seq, seq[1:]):
            if wl.direction == "max":
                assert a > c or (a == c and ia < ic)
            else:
                assert a < c or (a == c and ia < ic)
        # tie membership follows the tie-break at the boundary value
        if len(rest):
            worst = chosen.min() if wl.direction == "max" else chosen.max()
            ties_in = picks[chosen == worst]
            ties_out = rest[nums[rest] == worst]
            if len(ties_out):
                if wl.tie_break == "prefer_larger_index":
                    assert ties_in.min() > ties_out.max()
                else:
                    assert ties_in.max() < ties_out.min()
    if cfg in (1, 5):
        # -0.0 survives bitwise somewhere in the output
        negzero = {"f32": 0x80000000, "f64": 0x8000000000000000}[wl.dtype]
        assert np.any(wl.keys == negzero)


def test_untouched_tail_and_empty_segments():
    keys = W.f32_bits(np.array([3.0, 1.0, 2.0, 9.0, 8.0], dtype=np.float32))
    vals = np.arange(5, dtype=np.int32)
    # segment 0: [0,3); segment 1: empty (end < begin); segment 2: [3,5)
    offs = np.array([0, 3, 1, 5], dtype=np.int64)
    ok = np.full(3 * 4, 0xDEADBEEF, dtype=np.uint32)
    ov = np.full(3 * 4, -7, dtype=np.int32)
    oracle.batched_topk("f32", keys, vals, offs, 4, "max", "prefer_smaller_index", ok, ov)
    assert list(ov) == [0, 2, 1, -7, -7, -7, -7, -7, 3, 4, 2, 1]
    assert list(ok[3:8]) == [0xDEADBEEF] * 5
