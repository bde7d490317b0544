"""Fused LM-head projection + cross-entropy for GB300 (sm_103a).

The work runs in libflce.so (hand-written tcgen05/TMA kernels behind the C-ABI
declared in include/flce.h); this package is its Python binding. Importing it
fails when the library has not been built: there is no CPU fallback.
"""

from ._binding import (  # noqa: F401
    FLAG_COMPACT_IGNORED,
    FLAG_FILTER_FULL_DH,
    FLAG_FILTER_FULL_DW,
    FLAG_SORT_VOCAB,
    FLAG_TEST_SHORT_WAITS,
    REDUCTIONS,
    AdamwHparams,
    adamw_hparams_bytes,
    FlceError,
    FlceProblem,
    LaunchProfiler,
    Status,
    declared_symbols,
    flce_forward,
    flce_adamw_step,
    flce_backward_ex,
    flce_count_valid,
    flce_forward_backward,
    flce_forward_backward_global,
    flce_forward_backward_adamw,
    flce_forward_ex,
    flce_forward_static_scratch,
    flce_forward_workspace_bytes,
    flce_get_device_status,
    flce_get_filter_stats,
    flce_get_vocab_order,
    flce_status_string,
    flce_workspace_bytes,
    lib,
    make_problem,
)
from .api import (FusedAdamWHead, Workspace, adamw_hparams, device_status, forward,  # noqa: F401
                  forward_backward, forward_backward_adamw)
from .autograd import FusedLinearCrossEntropy, linear_cross_entropy  # noqa: F401
from .data_parallel import DataParallelStep, exchange_step  # noqa: F401
