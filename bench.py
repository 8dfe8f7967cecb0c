#!/usr/bin/env python
"""Benchmark of segmented top-k on GB300 (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 1..5|5det]

A step is one segmented top-k call over the whole batch of the workload
(default: workload 2, 128 segments x 152,064 fp32 keys ~ N(0,1), k = 50, max,
pairs with value = source index, gpu_to_gpu + prefer_smaller_index +
stable_sorted). `value` is keys/s over all ranks with the inputs already in
HBM; inputs rotate over enough copies that every step reads from HBM, not L2.
The timed steps are replayed from CUDA graphs of library calls, so host
launch overhead is not measured. `e2e` is the same metric through the
host-buffer entry point, host<->device copies included.

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

def workload_for(name: str):
    from segmented_radix_top_gb300 import workloads as W
    if name == "5det":
        return W.workload5(mode="det")
    if name == "5":
        return W.workload5(mode="nondet")
    return W.by_number(int(name))


def kernel_label(wl, launches: int, sms: int) -> str:
    """The kernels one step launches: with k <= 32 short segments take a
    warp-select kernel (one warp each with many segments, eight with few),
    longer ones the CTA / cluster kernel."""
    cta = "stream_topk_kernel<%s>" % wl.dtype
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
    wl = workload_for(args.workload)
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

def run_ours(args, ws, rank, local):
    import torch
    import segmented_radix_top_gb300 as st
    from segmented_radix_top_gb300 import workloads as W

    TORCH_VIEW = {"f16": torch.int16, "bf16": torch.int16, "f32": torch.int32, "f64": torch.int64,
                  "u32": torch.int32, "i32": torch.int32}
    NUMPY_SIGNED = {"f16": np.int16, "bf16": np.int16, "f32": np.int32, "f64": np.int64,
                    "u32": np.int32, "i32": np.int32}
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st.build()
    wl = workload_for(args.workload)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or L2_FALLBACK)

    keys_np = np.ascontiguousarray(wl.keys).view(NUMPY_SIGNED[wl.dtype])
    key_bytes = keys_np.nbytes
    copies = max(2, -(-3 * l2 // key_bytes))  # inputs of one rotation exceed 3x L2
    keys_d = [torch.from_numpy(keys_np).to(dev) for _ in range(copies)]
    vals_d = [torch.from_numpy(wl.values).to(dev) for _ in range(copies)] if wl.values is not None else None
    offs_d = torch.from_numpy(wl.offsets).to(dev)
    S, k = wl.num_segments, wl.k
    out_k = torch.empty(S * k, dtype=TORCH_VIEW[wl.dtype], device=dev)
    out_v = torch.empty(S * k, dtype=torch.int32, device=dev) if wl.values is not None else None
    ml = wl.max_segment_len
    n_keys = int(wl.lengths.sum())

    def call(i):
        st.batched_topk(keys_d[i % copies], offs_d, k, values=vals_d[i % copies] if vals_d else None,
                        key_dtype=wl.dtype, direction=wl.direction, determinism=wl.determinism,
                        tie_break=wl.tie_break, ordering=wl.ordering, out_keys=out_k,
                        out_values=out_v, max_segment_len=ml)

    # warm-up (eager): plans the launch, raises the shared-memory opt-in
    for i in range(max(args.warmup, 1)):
        call(i)
    torch.cuda.synchronize(dev)
    launches_per_step = st.last_launch_count()
    assert st.read_device_error() == 0

    # CUDA graphs of G consecutive steps (rotating over the input copies)
    G = max(1, min(args.steps, 64))
    s = torch.cuda.Stream(dev)
    graphs = {}

    def graph_for(n):
        if n not in graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    call(i)
            graphs[n] = g
        return graphs[n]

    full, rem = divmod(args.steps, G)
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
    with ClockSampler(local) as clk:
        e0.record(cur)
        for n in plan:
            graphs[n].replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    el = e0.elapsed_time(e1) / 1e3
    el_max = reduce_max(el, ws, dev)
    step_s = el_max / args.steps
    # device time of one step: one launch, or the warp-path launch for short
    # segments plus the CTA launch for the rest (their bytes are counted together)
    kernel_s = el / args.steps
    assert st.read_device_error() == 0

    # end to end through the host-buffer entry point (pinned host memory)
    h_keys = torch.from_numpy(keys_np).pin_memory()
    h_vals = torch.from_numpy(wl.values).pin_memory() if wl.values is not None else None
    h_offs = torch.from_numpy(wl.offsets).pin_memory()
    h_ok = torch.empty(S * k, dtype=TORCH_VIEW[wl.dtype]).pin_memory()
    h_ov = torch.empty(S * k, dtype=torch.int32).pin_memory() if h_vals is not None else None
    ws_bytes = st.host_workspace_bytes(wl.dtype, h_vals is not None, wl.num_keys, S, k)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    e2e_steps = max(1, min(args.steps, 30))

    def host_call():
        st.batched_topk_host(wl.dtype, h_keys, h_offs, k, workspace, values=h_vals,
                             direction=wl.direction, determinism=wl.determinism,
                             tie_break=wl.tie_break, ordering=wl.ordering, out_keys=h_ok,
                             out_values=h_ov, max_segment_len=ml)

    for _ in range(2):
        host_call()
    torch.cuda.synchronize(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_call()
    torch.cuda.synchronize(dev)
    e2e_el = reduce_max(time.perf_counter() - t0, ws, dev)
    h2d = h_keys.numel() * h_keys.element_size() + h_offs.numel() * 8 + \
        h_ok.numel() * h_ok.element_size()
    d2h = h_ok.numel() * h_ok.element_size()
    if h_vals is not None:
        h2d += h_vals.numel() * 4 + h_ov.numel() * 4
        d2h += h_ov.numel() * 4

    if rank != 0:
        return 0
    peak, peak_note = measured_peak()
    alg = algorithmic_bytes(wl)
    achieved = alg / kernel_s / 1e9
    cpu_value, cpu_desc = oracle_keys_per_s(wl, seconds=10.0, threads=os.cpu_count() or 1)
    workload_key = args.workload
    line = {
        "metric": METRIC,
        "value": ws * n_keys / step_s,
        "unit": "keys/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded PCG64 generators, segmented_radix_top_gb300/workloads.py)",
        "config": {"workload": wl.name, "segments": S, "keys": n_keys, "k": k,
                   "direction": wl.direction, "determinism": wl.determinism,
                   "tie_break": wl.tie_break, "ordering": wl.ordering,
                   "pairs": wl.values is not None,
                   "l2": "inputs rotate over %d copies (%.0f MB of keys) > L2 %.0f MB" % (
                       copies, copies * key_bytes / 1e6, l2 / 1e6),
                   "timing": "CUDA graphs of %d calls, CUDA events on the replay stream" % G},
        "segments_per_s": ws * S / step_s,
        "hbm_gbs": alg / kernel_s / 1e9,
        "formula_gbs": formula_bytes(wl) / kernel_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_note": peak_note,
                     "traffic": profiled_traffic(workload_key),
                     "algorithmic_bytes_per_launch": alg,
                     "launches_per_step": launches_per_step,
                     "kernel": kernel_label(wl, launches_per_step, props.multi_processor_count)},
        "cpu_baseline": {"value": cpu_value, "unit": "keys/s", "cores": os.cpu_count() or 1,
                         "kind": "oracle", "sample": cpu_desc},
        "e2e": {"value": ws * n_keys * e2e_steps / e2e_el, "unit": "keys/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="2", choices=["1", "2", "3", "4", "5", "5det"])
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
