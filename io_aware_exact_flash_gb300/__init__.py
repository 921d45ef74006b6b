"""Exact attention forward for GB300 (sm_103a): dense, paged/ragged prefill, split-KV decode and
the paged KV append that feeds them.

The compute path is the C-ABI library ``libfa_gb300.so`` (declared in ``include/fa.h``); this
package is its thin binding plus the seeded workload generator used by tests and benchmarks.
"""
from .binding import (  # noqa: F401
    EXPORTED,
    FaError,
    fa_cascade_fwd,
    fa_cascade_workspace_bytes,
    fa_decode_num_splits,
    fa_fwd,
    fa_get_device_status,
    fa_merge_states,
    fa_paged_append,
    fa_paged_decode_noalloc,
    fa_paged_fwd,
    fa_paged_num_splits,
    fa_selftest_wait_timeout,
    fa_paged_workspace_bytes,
    load_library,
    status_string,
)
from .buildlib import LIBRARY, build as build_library  # noqa: F401
