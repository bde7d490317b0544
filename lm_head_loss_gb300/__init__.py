"""Fused LM-head projection + cross-entropy for GB300 (sm_103a).

The work runs in libflce.so (hand-written tcgen05/TMA kernels behind the C-ABI
declared in include/flce.h); this package is its Python binding. Importing it
fails when the library has not been built: there is no CPU fallback.
"""

from ._binding import (  # noqa: F401
    FLAG_TEST_SHORT_WAITS,
    FlceError,
    FlceProblem,
    LaunchProfiler,
    Status,
    declared_symbols,
    flce_forward,
    flce_forward_backward,
    flce_forward_static_scratch,
    flce_get_device_status,
    flce_get_filter_stats,
    flce_status_string,
    flce_workspace_bytes,
    lib,
    make_problem,
)
from .api import Workspace, device_status, forward, forward_backward  # noqa: F401
