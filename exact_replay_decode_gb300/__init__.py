"""Exact-replay SSD for GB300: chunked Mamba2 SSD prefill, exact-replay decode, checkpoint refresh,
output-only speculative verify and commit, the causal conv1d upstream of the SSM, and a
per-token-writeback SSU comparison kernel, as a
C-ABI CUDA library (libers.so, include/ers.h) with a thin PyTorch binding.

Importing the package is cheap; the CUDA library is loaded on first use of an operation and its
absence is an error (there is no fallback path).
"""
__version__ = "0.1.0"

_OPS = ("LayerParams", "ReplayCache", "Status", "ssd_scan_fwd", "ssd_scan_fwd_static", "STATIC_SCRATCH_BYTES",
        "chunked_prefill", "replay_decode", "refresh",
        "spec_verify", "commit", "ssu_update", "conv1d_fwd", "conv1d_update", "GdnCache", "gdn_verify",
        "gdn_commit", "gdn_refresh", "selftest_bounded_wait", "spec_verify_exact", "commit_exact")


def __getattr__(name):
    if name in _OPS:
        from . import ops
        return getattr(ops, name)
    if name in ("ErsError",):
        from . import _abi
        return _abi.ErsError
    raise AttributeError(name)


__all__ = list(_OPS) + ["ErsError"]
