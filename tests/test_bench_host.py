"""Host-side pieces of bench.py: byte accounting and the max-over-ranks
timing reduction with two gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from segmented_radix_top_gb300 import workloads as W


def test_algorithmic_bytes_workload2():
    wl = W.workload2(segments=4, seg_len=1000)
    # 4000 fp32 keys read; 200 selected: 200 values read, 200 keys + 200 values written; 5 offsets
    assert bench.algorithmic_bytes(wl) == 4000 * 4 + 200 * (4 + 8) + 5 * 8
    assert bench.formula_bytes(wl) == 4000 * 8 + 200 * 8


def test_algorithmic_bytes_short_segments():
    wl = W.random_workload(1, "f64", [3, 0, 10], 5, pairs=False)
    assert bench.algorithmic_bytes(wl) == 13 * 8 + 8 * 8 + 4 * 8


def test_profiling_workloads_scale_the_segment_count():
    # bench.py --profile-calls N --segments S: the same workload shape with S
    # segments (the array workload: S keys), for captures of a smaller case
    wl = bench.workload_for("5det", 8)
    assert wl.num_segments == 8 and wl.k == 256 and wl.ordering == "stable_sorted"
    assert int(wl.lengths.min()) == int(wl.lengths.max()) == 32768
    wl = bench.workload_for("2", 3)
    assert wl.num_segments == 3 and int(wl.lengths.max()) == 152064 and wl.k == 50
    wl = bench.workload_for("array", 1 << 16)
    assert wl.info.get("array") and wl.num_keys == 1 << 16 and wl.k == 1024
    assert bench.workload_for("4", 2).num_segments == 2
    assert bench.workload_for("3", 50).num_segments == 50


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    # a committed capture counts only while the kernel sources hash the same
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.txt").write_text("bench_workload: 2\nsource_hash: %s\ndram_bytes_per_launch: 1234\n"
                                % bench.kernel_source_hash())
    (prof / "y.txt").write_text("bench_workload: 4\nsource_hash: 0000000000000000\ndram_bytes_per_launch: 99\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "segmented_radix_top_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in os.listdir(os.path.join(os.path.dirname(bench.__file__), "segmented_radix_top_gb300", "csrc")):
        full = os.path.join(os.path.dirname(bench.__file__), "segmented_radix_top_gb300", "csrc", name)
        if os.path.isfile(full):
            (src / name).write_bytes(open(full, "rb").read())
    assert bench.profiled_traffic("2") == 1234
    assert bench.profiled_traffic("4") is None      # taken with other sources
    assert bench.profiled_traffic("5det") is None   # no capture


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    out[rank] = bench.reduce_max(1.5 + rank, 2)
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 2.5 and out[1] == 2.5


def test_dist_setup_defaults(monkeypatch):
    for v in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
