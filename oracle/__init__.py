"""fp64 CPU oracle for the fused LM-head projection plus cross-entropy.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, links or calls this
package; only the test suite, the smoke check and the benchmark's CPU-baseline
arm use it. It shares no code with the CUDA path.
"""

from .flce_oracle import (  # noqa: F401
    IGNORE_INDEX,
    adamw_step,
    average_logits,
    dlogits,
    dH_rows,
    dW_rows,
    forward,
    forward_backward,
    forward_backward_adamw,
    forward_backward_ex,
    forward_backward_filtered,
    inputs_f64,
    logits,
    logsumexp_rows,
    loss_value,
    lse_rows,
    valid_count,
    vocabulary_order,
)
