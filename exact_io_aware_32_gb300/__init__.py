"""Exact, IO-aware scaled-dot-product attention for NVIDIA GB300 (sm_103a).

The kernels sit behind the C ABI of ``include/fa.h`` (``libfa.so``); this
package holds the thin ctypes binding (``fa``), the build script, the seeded
input generators and the flop/byte model the benchmark reports against.
"""
from .fa import (  # noqa: F401
    FA_OK, FAError, attention, backward, backward_dropout, backward_kv, fa_bwd, fa_bwd_dropout, fa_bwd_kv,
    fa_bwd_kv_workspace_bytes, fa_bwd_noalloc, fa_bwd_workspace_bytes, fa_device_status, fa_fwd, fa_fwd_dropout,
    fa_fwd_fp8, fa_fwd_kv, fa_fwd_kv_workspace_bytes, fa_status_string, fa_test_arm_fault, forward, forward_dropout,
    forward_fp8, forward_kv,
)
