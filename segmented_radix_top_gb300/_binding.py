"""ctypes binding of libsegtopk.so (argument marshalling only).

Every step of the selection runs in the library's CUDA kernels; this module
turns tensors into pointers and names into enum values. It never falls back
to another implementation: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

# Enum values of include/segtopk.h
DTYPE = {"f16": 0, "bf16": 1, "f32": 2, "f64": 3, "u32": 4, "i32": 5}
KEY_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "f64": 8, "u32": 4, "i32": 4}
DIRECTION = {"max": 0, "min": 1}
DETERMINISM = {"not_guaranteed": 0, "run_to_run": 1, "gpu_to_gpu": 2}
TIE_BREAK = {"unspecified": 0, "prefer_smaller_index": 1, "prefer_larger_index": 2}
ORDERING = {"unsorted": 0, "sorted": 1, "stable_sorted": 2}
STATUS = {0: "SUCCESS", 1: "INVALID_VALUE", 2: "INVALID_COMBINATION", 3: "NOT_SUPPORTED",
          4: "MISALIGNED", 5: "CUDA", 6: "DEVICE"}
MAX_K = 2048
NOALLOC_STAGING_BYTES = 32 * 1024 * 1024  # SEGTOPK_NOALLOC_STAGING_BYTES

_TORCH_TO_DTYPE = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32",
                   torch.float64: "f64", torch.int32: "i32"}
if hasattr(torch, "uint32"):
    _TORCH_TO_DTYPE[torch.uint32] = "u32"


class SegTopKError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status
        self.name = STATUS.get(status, str(status))


class Options(ctypes.Structure):
    _fields_ = [("cluster_width", ctypes.c_int32), ("small_segment_max_len", ctypes.c_int32),
                ("team_segment_max_len", ctypes.c_int32), ("reserved", ctypes.c_int32 * 5)]


_lib = None
_instr = None
STAT_NAMES = ["ctas", "cycles", "first_bound_cycles", "stream_cycles", "final_cycles", "chunks", "trims",
              "restreams", "list_entries", "sampled_bounds", "digit_passes", "wait_cycles_warp0", "keys",
              "candidate_shares_warp0", "overflowing_offers", "spec_warp_cycles", "spec_merge_cycles",
              "spec_keep_cycles", "final_select_cycles", "final_write_cycles", "select_pass_cycles",
              "select_finish_cycles", "select_compact_cycles"]


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libsegtopk.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = _open(_build.LIB_PATH)
    return _lib


def load_instrumented():
    """Load the instrumented build (statistics counters and test hooks),
    building it first if needed. Its calls are the same as load()'s."""
    global _instr
    if _instr is None:
        _instr = _open(_build.build(variant="instr"))
    return _instr


def _open(path):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built (run __graft_entry__.build()); "
                           "there is no fallback implementation" % os.path.basename(path))
    L = ctypes.CDLL(path)
    c_int, c_i32, c_i64, vp = ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    L.segtopk_batched_topk.restype = c_int
    L.segtopk_batched_topk.argtypes = [c_int, vp, vp, vp, c_i64, c_i32, c_int, c_int, c_int, c_int,
                                       vp, vp, c_i64, vp]
    L.segtopk_batched_topk_ex.restype = c_int
    L.segtopk_batched_topk_ex.argtypes = [c_int, vp, vp, vp, c_i64, c_i32, c_int, c_int, c_int, c_int,
                                          vp, vp, c_i64, ctypes.POINTER(Options), vp]
    L.segtopk_batched_topk_values.restype = c_int
    L.segtopk_batched_topk_values.argtypes = [c_int, vp, vp, c_i32, vp, c_i64, c_i32, c_int, c_int, c_int, c_int,
                                              vp, vp, c_i64, ctypes.POINTER(Options), vp]
    L.segtopk_topk.restype = c_int
    L.segtopk_topk.argtypes = [c_int, vp, vp, c_i32, c_i64, c_i32, c_int, c_int, c_int, c_int, vp, vp, vp,
                               ctypes.c_size_t, vp]
    L.segtopk_topk_workspace_bytes.restype = ctypes.c_size_t
    L.segtopk_topk_workspace_bytes.argtypes = [c_int, c_i32, c_i64, c_i32]
    L.segtopk_batched_topk_host.restype = c_int
    L.segtopk_batched_topk_host.argtypes = [c_int, vp, vp, vp, c_i64, c_i32, c_int, c_int, c_int,
                                            c_int, vp, vp, c_i64, vp, ctypes.c_size_t, vp]
    L.segtopk_batched_topk_host_noalloc.restype = c_int
    L.segtopk_batched_topk_host_noalloc.argtypes = [c_int, vp, vp, vp, c_i64, c_i32, c_int, c_int, c_int,
                                                    c_int, vp, vp, c_i64, vp]
    L.segtopk_host_workspace_bytes.restype = ctypes.c_size_t
    L.segtopk_host_workspace_bytes.argtypes = [c_int, c_int, c_i64, c_i64, c_i32]
    L.segtopk_status_string.restype = ctypes.c_char_p
    L.segtopk_status_string.argtypes = [c_int]
    L.segtopk_last_cuda_error.restype = c_int
    L.segtopk_last_cuda_error.argtypes = []
    L.segtopk_last_launch_count.restype = c_int
    L.segtopk_last_launch_count.argtypes = []
    L.segtopk_read_device_error.restype = c_int
    L.segtopk_read_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.segtopk_read_stats.restype = c_int
    L.segtopk_read_stats.argtypes = [ctypes.POINTER(ctypes.c_uint64), c_int]
    L.segtopk_set_test_hooks.restype = c_int
    L.segtopk_set_test_hooks.argtypes = [ctypes.c_longlong, ctypes.c_uint32]
    L.segtopk_test_device_prep.restype = c_int
    L.segtopk_test_device_prep.argtypes = [c_int, ctypes.POINTER(c_int), ctypes.POINTER(ctypes.c_uint32),
                                           ctypes.POINTER(c_int), ctypes.POINTER(ctypes.c_uint32)]
    return L


def _check(rc: int, lib=None):
    if rc != 0:
        L = lib if lib is not None else load()
        msg = L.segtopk_status_string(rc).decode()
        if rc == 5:
            msg += " (cudaError %d)" % L.segtopk_last_cuda_error()
        raise SegTopKError(rc, "segtopk: " + msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def key_dtype_of(t: torch.Tensor, key_dtype: str | None) -> str:
    if key_dtype is not None:
        if t.element_size() != KEY_BYTES[key_dtype]:
            raise ValueError("keys element size does not match key_dtype %s" % key_dtype)
        return key_dtype
    if t.dtype not in _TORCH_TO_DTYPE:
        raise ValueError("cannot infer key type from %s; pass key_dtype" % t.dtype)
    return _TORCH_TO_DTYPE[t.dtype]


def batched_topk(keys: torch.Tensor, segment_offsets: torch.Tensor, k: int, *, values=None,
                 direction: str = "max", determinism: str = "gpu_to_gpu",
                 tie_break: str = "prefer_smaller_index", ordering: str = "stable_sorted",
                 out_keys=None, out_values=None, max_segment_len: int | None = None,
                 key_dtype: str | None = None, stream=None, cluster_width: int = 0,
                 small_segment_max_len: int = 0, team_segment_max_len: int = 0, lib=None):
    """Segmented top-k on the GPU through libsegtopk (see include/segtopk.h).

    keys: 1-D CUDA tensor (any view; its data pointer aligned to the element
    size); its element size must match the key type (a raw-bits tensor of
    the same width works with key_dtype).
    segment_offsets: int64 CUDA tensor of num_segments + 1 offsets.
    values: optional int32 or int64 CUDA tensor parallel to keys (int64
    values take segtopk_batched_topk_values).
    Returns (out_keys, out_values) of shape [num_segments * k]; out_values is
    None for keys-only calls. Slots past a short segment's length are left as
    they were in the given out tensors (uninitialised if allocated here).
    cluster_width forces the CTAs per segment (0: automatic);
    small_segment_max_len / team_segment_max_len set which segments take one
    warp / a team of eight warps each when k <= 32 (0: the defaults, or none
    with a forced width; < 0: none). `lib` selects another build of the
    library (load_instrumented()).
    """
    L = lib if lib is not None else load()
    kd = key_dtype_of(keys, key_dtype)
    if segment_offsets.dtype != torch.int64:
        raise ValueError("segment_offsets must be int64")
    num_segments = segment_offsets.numel() - 1
    if out_keys is None:
        out_keys = torch.empty(max(num_segments, 0) * k, dtype=keys.dtype, device=keys.device)
    wide = values is not None and values.dtype == torch.int64
    if values is not None and values.dtype not in (torch.int32, torch.int64):
        raise ValueError("values must be int32 or int64")
    if values is not None and out_values is None:
        out_values = torch.empty(max(num_segments, 0) * k, dtype=values.dtype, device=keys.device)
    if values is not None and out_values.dtype != values.dtype:
        raise ValueError("out_values must have the dtype of values")
    ml = -1 if max_segment_len is None else int(max_segment_len)
    opts = Options()
    opts.cluster_width = int(cluster_width)
    opts.small_segment_max_len = int(small_segment_max_len)
    opts.team_segment_max_len = int(team_segment_max_len)
    if wide:
        rc = L.segtopk_batched_topk_values(DTYPE[kd], _ptr(keys), _ptr(values), 8, _ptr(segment_offsets),
                                           num_segments, int(k), DIRECTION[direction],
                                           DETERMINISM[determinism], TIE_BREAK[tie_break], ORDERING[ordering],
                                           _ptr(out_keys), _ptr(out_values), ml, ctypes.byref(opts),
                                           _stream_handle(stream, keys.device))
    else:
        rc = L.segtopk_batched_topk_ex(DTYPE[kd], _ptr(keys), _ptr(values), _ptr(segment_offsets),
                                       num_segments, int(k), DIRECTION[direction],
                                       DETERMINISM[determinism], TIE_BREAK[tie_break], ORDERING[ordering],
                                       _ptr(out_keys), _ptr(out_values), ml, ctypes.byref(opts),
                                       _stream_handle(stream, keys.device))
    _check(rc, L)
    return out_keys, out_values


def topk(keys: torch.Tensor, k: int, *, values=None, direction: str = "max",
         determinism: str = "gpu_to_gpu", tie_break: str = "prefer_smaller_index",
         ordering: str = "stable_sorted", out_keys=None, out_values=None, key_dtype: str | None = None,
         workspace=None, stream=None, lib=None):
    """Top-k over one array (segtopk_topk): keys is a 1-D CUDA tensor,
    values an optional int32 / int64 tensor of the same length. The device
    workspace is allocated here (as a torch tensor) unless given.
    Returns (out_keys, out_values) of k slots (out_values None for keys only)."""
    L = lib if lib is not None else load()
    kd = key_dtype_of(keys, key_dtype)
    n = keys.numel()
    vb = 0 if values is None else values.element_size()
    if values is not None and values.dtype not in (torch.int32, torch.int64):
        raise ValueError("values must be int32 or int64")
    if out_keys is None:
        out_keys = torch.empty(k, dtype=keys.dtype, device=keys.device)
    if values is not None and out_values is None:
        out_values = torch.empty(k, dtype=values.dtype, device=keys.device)
    need = int(L.segtopk_topk_workspace_bytes(DTYPE[kd], vb, n, int(k)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=keys.device)
    rc = L.segtopk_topk(DTYPE[kd], _ptr(keys), _ptr(values), vb if vb else 4, n, int(k), DIRECTION[direction],
                        DETERMINISM[determinism], TIE_BREAK[tie_break], ORDERING[ordering], _ptr(out_keys),
                        _ptr(out_values), _ptr(workspace), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream, keys.device))
    _check(rc, L)
    return out_keys, out_values


def host_workspace_bytes(key_dtype: str, has_values: bool, num_keys: int, num_segments: int,
                         k: int) -> int:
    return int(load().segtopk_host_workspace_bytes(DTYPE[key_dtype], int(has_values), num_keys,
                                                   num_segments, k))


def batched_topk_host(key_dtype: str, keys: torch.Tensor, segment_offsets: torch.Tensor, k: int,
                      workspace: torch.Tensor, *, values=None, direction: str = "max",
                      determinism: str = "gpu_to_gpu", tie_break: str = "prefer_smaller_index",
                      ordering: str = "stable_sorted", out_keys=None, out_values=None,
                      max_segment_len: int | None = None, stream=None):
    """Host-buffer variant: keys/values/offsets/outputs are CPU tensors
    (pinned for full copy bandwidth); `workspace` is a CUDA byte tensor of at
    least host_workspace_bytes(...) bytes. Synchronises before returning."""
    L = load()
    num_segments = segment_offsets.numel() - 1
    if out_keys is None:
        out_keys = torch.empty(num_segments * k, dtype=keys.dtype)
    if values is not None and out_values is None:
        out_values = torch.empty(num_segments * k, dtype=torch.int32)
    ml = -1 if max_segment_len is None else int(max_segment_len)
    rc = L.segtopk_batched_topk_host(DTYPE[key_dtype], _ptr(keys), _ptr(values), _ptr(segment_offsets),
                                     num_segments, int(k), DIRECTION[direction],
                                     DETERMINISM[determinism], TIE_BREAK[tie_break],
                                     ORDERING[ordering], _ptr(out_keys), _ptr(out_values), ml,
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream, workspace.device))
    _check(rc)
    return out_keys, out_values


def batched_topk_host_noalloc(key_dtype: str, keys: torch.Tensor, segment_offsets: torch.Tensor, k: int, *,
                              values=None, direction: str = "max", determinism: str = "gpu_to_gpu",
                              tie_break: str = "prefer_smaller_index", ordering: str = "stable_sorted",
                              out_keys=None, out_values=None, max_segment_len: int | None = None,
                              stream=None, device=None):
    """Host-buffer variant that allocates no device memory: the library stages
    the call in its own fixed device array of NOALLOC_STAGING_BYTES (for
    callers that cannot allocate). Runs on the current CUDA device (or
    `device`); synchronises before returning; calls must not overlap."""
    L = load()
    num_segments = segment_offsets.numel() - 1
    if out_keys is None:
        out_keys = torch.empty(num_segments * k, dtype=keys.dtype)
    if values is not None and out_values is None:
        out_values = torch.empty(num_segments * k, dtype=torch.int32)
    ml = -1 if max_segment_len is None else int(max_segment_len)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    rc = L.segtopk_batched_topk_host_noalloc(DTYPE[key_dtype], _ptr(keys), _ptr(values), _ptr(segment_offsets),
                                             num_segments, int(k), DIRECTION[direction],
                                             DETERMINISM[determinism], TIE_BREAK[tie_break],
                                             ORDERING[ordering], _ptr(out_keys), _ptr(out_values), ml,
                                             _stream_handle(stream, dev))
    _check(rc)
    return out_keys, out_values


def read_device_error(lib=None) -> int:
    """Reads and clears the kernels' device error word (synchronises)."""
    w = ctypes.c_uint32(0)
    L = lib if lib is not None else load()
    _check(L.segtopk_read_device_error(ctypes.byref(w)), L)
    return int(w.value)


def read_stats() -> dict:
    """Sums and clears the instrumented build's per-CTA counters (synchronises)."""
    L = load_instrumented()
    arr = (ctypes.c_uint64 * len(STAT_NAMES))()
    _check(L.segtopk_read_stats(arr, len(STAT_NAMES)), L)
    return {name: int(arr[i]) for i, name in enumerate(STAT_NAMES)}


def set_test_hooks(wait_limit_cycles: int, first_copy_extra_bytes: int = 0):
    """Instrumented build only: the copy-wait bound and the bytes added to
    every slice's first copy's expected count (see include/segtopk.h)."""
    L = load_instrumented()
    _check(L.segtopk_set_test_hooks(int(wait_limit_cycles), int(first_copy_extra_bytes)), L)


def test_device_prep(launches):
    """Instrumented build only, no CUDA call: the attribute calls each of a
    sequence of launches (device, dynamic shared-memory bytes, cluster
    width; width <= 0 for the warp kernel) would make, per the library's
    per-device records (bit 0 opt-in, bit 1 wide clusters, bit 2 carveout;
    see include/segtopk.h)."""
    L = load_instrumented()
    n = len(launches)
    devs = (ctypes.c_int * max(n, 1))(*[int(d) for d, _, _ in launches])
    smem = (ctypes.c_uint32 * max(n, 1))(*[int(b) for _, b, _ in launches])
    cl = (ctypes.c_int * max(n, 1))(*[int(c) for _, _, c in launches])
    out = (ctypes.c_uint32 * max(n, 1))()
    _check(L.segtopk_test_device_prep(n, devs, smem, cl, out), L)
    return [int(out[i]) for i in range(n)]


def last_launch_count() -> int:
    return int(load().segtopk_last_launch_count())
