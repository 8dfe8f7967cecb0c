"""GB300-native segmented (batched) top-k by multi-pass radix digit selection.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
include/segtopk.h (libsegtopk.so); this package only marshals tensors into
that ABI (see _binding.py) and provides the seeded synthetic workloads
(workloads.py).
"""
from ._binding import (DETERMINISM, DIRECTION, DTYPE, KEY_BYTES, MAX_K, NOALLOC_STAGING_BYTES,  # noqa: F401
                       ORDERING, TIE_BREAK, SegTopKError, batched_topk, batched_topk_host,
                       batched_topk_host_noalloc, host_workspace_bytes,
                       last_launch_count, library_path, load, load_instrumented, read_device_error,
                       read_stats, set_test_hooks, topk)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libsegtopk.so for sm_103a in-tree (nvcc; no GPU needed)."""
    from . import _build
    return _build.build(force=force, verbose=verbose)
