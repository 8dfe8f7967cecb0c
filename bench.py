#!/usr/bin/env python
"""Benchmark of segmented top-k on GB300 (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 1..5|5det]

A step is one segmented top-k call over the whole batch of a workload. With
no --workload every workload is timed in turn (1, 2, 3, 4, 5 and 5det) and
`per_config` holds each one's line; the headline `value` is workload 5 in
its deterministic mode (4096 segments x 32,768 f64 keys, k = 256, max,
gpu_to_gpu + stable_sorted), the largest configuration. `value` is keys/s
over all ranks with the inputs already in HBM; inputs rotate over enough
copies that every step reads from HBM, not L2. The timed steps are replayed
from CUDA graphs of library calls, so host launch overhead is not measured.
`e2e` is the same metric through the host-buffer entry point,
host<->device copies included.

--stats prints the per-CTA counters of the instrumented build instead.

--impl reference times the CPU oracle (the only reference this subject has)
on this machine's host cores, on bounded samples of the same workload.
Multi-GPU (torchrun): every rank runs the same workload on its own GPU (weak
scaling); no collective touches the data path.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import glob
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "segments/sec and keys/sec per config; achieved HBM GB/s vs GB300 peak (1 GPU)"
L2_FALLBACK = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
# automatic warp-select limits (k <= 32): single warps up to 4096 keys with at
# least one segment per SM, teams of eight warps up to 8192 keys with fewer
SMALL_SEGMENT_DEFAULT = 4096
TEAM_SEGMENT_FEW = 8192


# ----------------------------------------------------------------------------- helpers

def workload_for(name: str, segments=None):
    """A benchmark workload; `segments` shrinks (or grows) its segment count
    (for the array workload: its key count), for profiling captures."""
    from segmented_radix_top_gb300 import workloads as W
    kw = {} if segments is None else {"segments": int(segments)}
    if name == "5det":
        return W.workload5(mode="det", **kw)
    if name == "5":
        return W.workload5(mode="nondet", **kw)
    if name == "array":
        return W.array_workload(**({} if segments is None else {"n": int(segments)}))
    if segments is not None:
        return {"1": W.workload1, "2": W.workload2, "3": W.workload3, "4": W.workload4}[name](**kw)
    return W.by_number(int(name))


def kernel_label(wl, launches: int, sms: int) -> str:
    """The kernels one step launches: with k <= 32 short segments take a
    warp-select kernel (one warp each with many segments, eight with few),
    longer ones the CTA / cluster kernel."""
    cta = "stream_topk_kernel<%s>" % wl.dtype
    if wl.info.get("array"):
        return "fill_piece_offsets + %s (pass 1, pieces) + %s (pass 2, candidates)" % (cta, cta)
    if wl.k > 32:
        return cta
    few = wl.num_segments < sms
    warp = "warp_topk_kernel<%s, %d warps>" % (wl.dtype, 8 if few else 1)
    limit = TEAM_SEGMENT_FEW if few else SMALL_SEGMENT_DEFAULT
    if int(wl.lengths.max()) <= limit:
        return warp
    if int(wl.lengths.min()) <= limit and launches == 2:
        return warp + " + " + cta + " (one step)"
    return cta


def algorithmic_bytes(wl) -> int:
    """Bytes one call must move: every key read once, the selected values read,
    the selected keys (and values) written, and the offsets read."""
    from segmented_radix_top_gb300 import workloads as W
    kb = W.KEY_BYTES[wl.dtype]
    n = int(wl.lengths.sum())
    m = int(np.minimum(wl.lengths, wl.k).sum())
    pairs = wl.values is not None
    return n * kb + m * (kb + (8 if pairs else 0)) + 8 * (wl.num_segments + 1)


def formula_bytes(wl) -> int:
    """Bytes of the target formula: keys (+ values) read once plus output written."""
    from segmented_radix_top_gb300 import workloads as W
    kb = W.KEY_BYTES[wl.dtype] + (4 if wl.values is not None else 0)
    n = int(wl.lengths.sum())
    m = int(np.minimum(wl.lengths, wl.k).sum())
    return n * kb + m * kb


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback (6.8 TB/s)"


def kernel_source_hash() -> str:
    """Hash of the CUDA sources with comments and whitespace removed, so that
    a profile taken with them stays valid across comment-only edits."""
    import re
    h = hashlib.sha1()
    for p in sorted(glob.glob(os.path.join(ROOT, "segmented_radix_top_gb300", "csrc", "*"))):
        with open(p, encoding="utf-8", errors="replace") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(os.path.basename(p).encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken with the current kernel sources; else None."""
    src = kernel_source_hash()
    for p in glob.glob(os.path.join(ROOT, "profiles", "*.txt")):
        kv = {}
        with open(p) as f:
            for line in f:
                if ":" in line and not line.startswith(" "):
                    a, b = line.split(":", 1)
                    kv[a.strip()] = b.strip()
        if kv.get("bench_workload") == workload and kv.get("source_hash") == src \
                and "dram_bytes_per_launch" in kv:
            try:
                return int(float(kv["dram_bytes_per_launch"]))
            except ValueError:
                return None
    return None


class ClockSampler:
    """SM clock and clock-event reasons sampled through NVML during a region."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self.period, self._stop, self._t, self.error = period_s, threading.Event(), None, None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            assert self.nvml.nvmlInit_v2() == 0
            self.h = ctypes.c_void_p()
            bus = None
            try:
                import torch
                p = torch.cuda.get_device_properties(cuda_index)
                bus = "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            except Exception:
                bus = None
            ok = False
            if bus is not None:
                ok = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
            if not ok:
                assert self.nvml.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) == 0
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self._reason_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception as e:  # sampling is best effort; the JSON says so
            self.nvml, self.error = None, repr(e)

    def _sample(self):
        mhz, r = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
            self.samples.append(int(mhz.value))
        if self._reason_fn(self.h, ctypes.byref(r)) == 0:
            self.reasons |= int(r.value)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def __enter__(self):
        if self.nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._t is not None:
            self._stop.set()
            self._t.join()
            self._sample()

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "error": self.error}
        names = [v for b, v in self.REASONS.items() if self.reasons & b and b != 0x1]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int, device=None) -> float:
    """Max over ranks (host-side timing only; never on the data path)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_keys_per_s(wl, seconds: float, threads: int):
    """The oracle as it stands, over passes of a bounded sample of the workload
    (whole segments, spread over `threads` host threads), for `seconds`."""
    import oracle
    lens = wl.lengths
    # the sample: the first segments holding about 8M keys (all of them if fewer)
    csum = np.cumsum(lens)
    nseg = int(np.searchsorted(csum, 8_000_000)) + 1
    nseg = min(max(nseg, 1), wl.num_segments)
    offs = wl.offsets[: nseg + 1]
    keys_in = int(np.maximum(np.diff(offs), 0).sum())
    out_k = np.zeros(nseg * wl.k, dtype=wl.keys.dtype)
    out_v = np.zeros(nseg * wl.k, dtype=np.int32) if wl.values is not None else None
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.batched_topk(wl.dtype, wl.keys, wl.values, offs, wl.k, wl.direction, wl.tie_break,
                            out_keys=out_k, out_values=out_v, threads=threads)
        done += keys_in
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done / el, "%d of %d segments (%d keys), repeated for %.1f s" % (
        nseg, wl.num_segments, keys_in, el)


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    wl = workload_for(args.workload or HEADLINE)
    threads = os.cpu_count() or 1
    # each step: `threads` segments of the workload (truncated to sample_len
    # keys) sorted in parallel; the sample is sized so the run stays short
    lens = wl.lengths
    sample_len = int(min(lens.max(), 1 << 20))
    seg_ids = np.argsort(-lens, kind="stable")[:threads]

    def make_sample(L):
        parts, offs = [], [0]
        vals = [] if wl.values is not None else None
        for s in seg_ids:
            b = int(wl.offsets[s]); n = int(min(lens[s], L))
            parts.append(wl.keys[b:b + n])
            if vals is not None:
                vals.append(wl.values[b:b + n])
            offs.append(offs[-1] + n)
        return (np.concatenate(parts), np.concatenate(vals) if vals is not None else None,
                np.array(offs, dtype=np.int64))

    def step(sample):
        k_, v_, o_ = sample
        oracle.batched_topk(wl.dtype, k_, v_, o_, wl.k, wl.direction, wl.tie_break, threads=threads)

    sample = make_sample(sample_len)
    t0 = time.perf_counter(); step(sample); one = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)
    while one > budget and sample_len > 256:
        sample_len //= 2
        sample = make_sample(sample_len)
        t0 = time.perf_counter(); step(sample); one = time.perf_counter() - t0
    for _ in range(args.warmup):
        step(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(sample)
    el = time.perf_counter() - t0
    keys_per_step = int(sample[2][-1])
    value = keys_per_step * args.steps / el
    desc = "%d segments x <=%d keys per step (the longest segments of the workload)" % (
        len(seg_ids), sample_len)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "keys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name},
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

TORCH_VIEW_NAMES = {"f16": "int16", "bf16": "int16", "f32": "int32", "f64": "int64", "u32": "int32", "i32": "int32"}
NUMPY_SIGNED = {"f16": np.int16, "bf16": np.int16, "f32": np.int32, "f64": np.int64, "u32": np.int32,
                "i32": np.int32}
# every workload of a default run (5: not_guaranteed + unsorted, 5det: gpu_to_gpu + stable_sorted);
# the headline is the largest configuration in its deterministic mode
ALL_WORKLOADS = ["1", "2", "3", "4", "5", "5det", "array"]
HEADLINE = "5det"


class Resident:
    """A workload's inputs in HBM, rotated over enough copies that one
    rotation exceeds 3 x L2 (every step reads from HBM, not L2)."""

    def __init__(self, wl, dev, l2):
        import torch
        self.wl = wl
        keys_np = np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])
        self.key_bytes = keys_np.nbytes
        self.copies = max(2, -(-3 * l2 // max(self.key_bytes, 1)))
        self.keys = [torch.from_numpy(keys_np).to(dev) for _ in range(self.copies)]
        self.vals = [torch.from_numpy(wl.values).to(dev) for _ in range(self.copies)] \
            if wl.values is not None else None
        self.offs = torch.from_numpy(wl.offsets).to(dev)
        tv = getattr(torch, TORCH_VIEW_NAMES[wl.dtype])
        self.out_k = torch.empty(wl.num_segments * wl.k, dtype=tv, device=dev)
        self.out_v = torch.empty(wl.num_segments * wl.k, dtype=torch.int32, device=dev) \
            if wl.values is not None else None
        self.array = bool(wl.info.get("array"))
        if self.array:
            import segmented_radix_top_gb300 as st
            need = st.load().segtopk_topk_workspace_bytes(st.DTYPE[wl.dtype], 4 if wl.values is not None else 0,
                                                          wl.num_keys, wl.k)
            self.workspace = torch.empty(max(int(need), 256), dtype=torch.uint8, device=dev)

    def call(self, i, lib=None):
        import segmented_radix_top_gb300 as st
        wl = self.wl
        if self.array:
            st.topk(self.keys[i % self.copies], wl.k, values=self.vals[i % self.copies] if self.vals else None,
                    key_dtype=wl.dtype, direction=wl.direction, determinism=wl.determinism,
                    tie_break=wl.tie_break, ordering=wl.ordering, out_keys=self.out_k, out_values=self.out_v,
                    workspace=self.workspace, lib=lib)
            return
        st.batched_topk(self.keys[i % self.copies], self.offs, wl.k,
                        values=self.vals[i % self.copies] if self.vals else None, key_dtype=wl.dtype,
                        direction=wl.direction, determinism=wl.determinism, tie_break=wl.tie_break,
                        ordering=wl.ordering, out_keys=self.out_k, out_values=self.out_v,
                        max_segment_len=wl.max_segment_len, lib=lib)


def time_device(res, steps, warmup, dev, ws):
    """Seconds per step over `steps` graph-replayed calls (CUDA events on the
    replay stream, a barrier and a synchronize on both sides, max over
    ranks), the launches per call, and the clocks sampled meanwhile."""
    import torch
    import segmented_radix_top_gb300 as st
    for i in range(max(warmup, 1)):  # eager: plans the launch, raises the shared-memory opt-in
        res.call(i)
    torch.cuda.synchronize(dev)
    launches = st.last_launch_count()
    assert st.read_device_error() == 0
    G = max(1, min(steps, 64))
    s = torch.cuda.Stream(dev)
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    res.call(i)
            graphs[n] = g
        return graphs[n]

    full, rem = divmod(steps, G)
    plan = [G] * full + ([rem] if rem else [])
    for n in set(plan):
        graph_for(n).replay()
    torch.cuda.synchronize(dev)
    for _ in range(2):  # warm replays
        for n in plan[:2]:
            graphs[n].replay()
    torch.cuda.synchronize(dev)
    cur = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        e0.record(cur)
        for n in plan:
            graphs[n].replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    el = e0.elapsed_time(e1) / 1e3
    assert st.read_device_error() == 0
    return reduce_max(el, ws, dev) / steps, el / steps, launches, clk.summary(), G


def time_e2e(wl, steps, dev, ws):
    """Keys per second through segtopk_batched_topk_host from pinned host
    buffers (host<->device copies inside the timed region), and the bytes
    copied per step."""
    import torch
    import segmented_radix_top_gb300 as st
    keys_np = np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])
    tv = getattr(torch, TORCH_VIEW_NAMES[wl.dtype])
    h_keys = torch.from_numpy(keys_np).pin_memory()
    h_vals = torch.from_numpy(wl.values).pin_memory() if wl.values is not None else None
    h_offs = torch.from_numpy(wl.offsets).pin_memory()
    S, k = wl.num_segments, wl.k
    h_ok = torch.empty(S * k, dtype=tv).pin_memory()
    h_ov = torch.empty(S * k, dtype=torch.int32).pin_memory() if h_vals is not None else None
    workspace = torch.empty(st.host_workspace_bytes(wl.dtype, h_vals is not None, wl.num_keys, S, k),
                            dtype=torch.uint8, device=dev)

    def host_call():
        st.batched_topk_host(wl.dtype, h_keys, h_offs, k, workspace, values=h_vals, direction=wl.direction,
                             determinism=wl.determinism, tie_break=wl.tie_break, ordering=wl.ordering,
                             out_keys=h_ok, out_values=h_ov, max_segment_len=wl.max_segment_len)

    for _ in range(2):
        host_call()
    torch.cuda.synchronize(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        host_call()
    torch.cuda.synchronize(dev)
    el = reduce_max(time.perf_counter() - t0, ws, dev)
    # keys, offsets and the output slots go to the device; keys and, for
    # pairs, the selected source indices come back (values stay on the host)
    h2d = h_keys.numel() * h_keys.element_size() + h_offs.numel() * 8 + h_ok.numel() * h_ok.element_size()
    d2h = h_ok.numel() * h_ok.element_size()
    if h_vals is not None:
        h2d += h_ov.numel() * 4
        d2h += h_ov.numel() * 4
    del workspace
    return ws * int(wl.lengths.sum()) * steps / el, h2d, d2h, steps


def config_line(name, wl, step_s, kernel_s, launches, clocks, G, copies, key_bytes, l2, sms, ws, steps):
    peak, peak_note = measured_peak()
    alg = algorithmic_bytes(wl)
    achieved = alg / kernel_s / 1e9
    n_keys = int(wl.lengths.sum())
    return {
        "workload": wl.name, "dtype": wl.dtype, "segments": wl.num_segments, "keys": n_keys, "k": wl.k,
        "direction": wl.direction, "determinism": wl.determinism, "tie_break": wl.tie_break,
        "ordering": wl.ordering, "pairs": wl.values is not None,
        "us_per_step": step_s * 1e6,
        "keys_per_s": ws * n_keys / step_s,
        "segments_per_s": ws * wl.num_segments / step_s,
        "hbm_gbs": achieved,
        "formula_gbs": formula_bytes(wl) / kernel_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_note": peak_note,
                     "traffic": profiled_traffic(name),
                     "algorithmic_bytes_per_launch": alg, "launches_per_step": launches,
                     "kernel": kernel_label(wl, launches, sms)},
        "gpu_launches": steps * launches,
        "l2": "inputs rotate over %d copies (%.0f MB of keys) > L2 %.0f MB" % (copies, copies * key_bytes / 1e6,
                                                                             l2 / 1e6),
        "timing": "CUDA graphs of %d calls, CUDA events on the replay stream" % G,
        "clocks": clocks,
    }


def run_ours(args, ws, rank, local):
    import torch
    import segmented_radix_top_gb300 as st
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st.build()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK)
    names = [args.workload] if args.workload else ALL_WORKLOADS
    headline = args.workload or HEADLINE
    per = {}
    head = None
    for name in names:
        wl = workload_for(name)
        res = Resident(wl, dev, l2)
        step_s, kernel_s, launches, clocks, G = time_device(res, args.steps, args.warmup, dev, ws)
        line = config_line(name, wl, step_s, kernel_s, launches, clocks, G, res.copies, res.key_bytes, l2,
                           props.multi_processor_count, ws, args.steps)
        del res
        torch.cuda.empty_cache()
        if wl.info.get("array"):
            line["e2e"] = None  # the single-array entry point takes device buffers only
        else:
            e2e_steps = max(1, min(args.steps, 10 if name == headline else 3))
            e2e_v, h2d, d2h, e2e_n = time_e2e(wl, e2e_steps, dev, ws)
            line["e2e"] = {"value": e2e_v, "unit": "keys/s", "h2d_bytes_per_step": h2d,
                           "d2h_bytes_per_step": d2h, "steps": e2e_n}
        torch.cuda.empty_cache()
        per[name] = line
        if name == headline:
            head = (wl, line)
    if rank != 0:
        return 0
    wl, hl = head
    threads = os.cpu_count() or 1
    cpu_value, cpu_desc = oracle_keys_per_s(wl, seconds=8.0, threads=threads)
    cpu_single, _ = oracle_keys_per_s(wl, seconds=6.0, threads=1)
    line = {
        "metric": METRIC,
        "value": hl["keys_per_s"],
        "unit": "keys/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": hl["us_per_step"] / 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded PCG64 generators, segmented_radix_top_gb300/workloads.py)",
        "config": {"workload": wl.name, "segments": wl.num_segments, "keys": hl["keys"], "k": wl.k,
                   "direction": wl.direction, "determinism": wl.determinism, "tie_break": wl.tie_break,
                   "ordering": wl.ordering, "pairs": wl.values is not None, "l2": hl["l2"],
                   "timing": hl["timing"]},
        "segments_per_s": hl["segments_per_s"],
        "hbm_gbs": hl["hbm_gbs"],
        "formula_gbs": hl["formula_gbs"],
        "roofline": hl["roofline"],
        "cpu_baseline": {"value": cpu_value, "unit": "keys/s", "cores": threads, "kind": "oracle",
                         "sample": cpu_desc, "single_thread_value": cpu_single},
        "e2e": hl["e2e"],
        "gpu_launches": hl["gpu_launches"],
        "clocks": hl["clocks"],
        "per_config": {n: {k: v for k, v in d.items() if k not in ("clocks",)} | {"sm_mhz": d["clocks"]["sm_mhz"]}
                       for n, d in per.items()},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_stats(args):
    """Per-CTA counters of the segment kernel (instrumented build) for each
    workload: one call after warm-up, summed over the launch's CTAs and
    averaged per CTA. Prints one JSON line."""
    import torch
    import segmented_radix_top_gb300 as st
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L = st.load_instrumented()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK)
    out = {}
    for name in ([args.workload] if args.workload else ALL_WORKLOADS):
        wl = workload_for(name)
        res = Resident(wl, dev, l2)
        for i in range(3):
            res.call(i, lib=L)
        torch.cuda.synchronize(dev)
        st.read_stats()
        res.call(0, lib=L)
        s = st.read_stats()
        ctas = max(s["ctas"], 1)
        per_cta = {k: round(v / ctas, 1) for k, v in s.items() if k != "ctas"}
        out[name] = {"workload": wl.name, "ctas": s["ctas"], "per_cta": per_cta}
        assert st.read_device_error(lib=L) == 0
        del res
        torch.cuda.empty_cache()
    print(json.dumps({"stats": out, "build": "libsegtopk_instr.so (SEGTOPK_STATS)"}), flush=True)
    return 0


def run_profile(args):
    """Plain (eager) calls of one workload, for ncu captures: no graphs, no
    host-buffer leg, no CPU baseline. Prints one line and exits."""
    import torch
    import segmented_radix_top_gb300 as st
    name = args.workload or HEADLINE
    wl = workload_for(name, args.segments)
    dev = torch.device("cuda", 0)
    res = Resident(wl, dev, 0)
    for i in range(args.profile_calls):
        res.call(i)
    torch.cuda.synchronize(dev)
    assert st.read_device_error() == 0
    print(json.dumps({"profile": name, "workload": wl.name, "calls": args.profile_calls,
                      "launches_per_call": st.last_launch_count(), "keys": int(wl.lengths.sum())}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=ALL_WORKLOADS,
                    help="time one workload only (default: all, workload 5 deterministic as the headline)")
    ap.add_argument("--stats", action="store_true",
                    help="print per-CTA counters of the instrumented build instead of timing")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="make this many plain calls of one workload and exit (ncu captures)")
    ap.add_argument("--segments", type=int, default=None,
                    help="with --profile-calls: the workload's segment count (array: key count)")
    args = ap.parse_args()
    if args.profile_calls > 0:
        return run_profile(args)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.stats:
        return run_stats(args) if rank == 0 else 0
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
