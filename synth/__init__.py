"""Seeded synthetic inputs for the fused LM-head cross-entropy.

This package draws the hidden states H, the LM-head weight W and the targets
y that both the fp64 oracle (``oracle/``) and the CUDA library are fed. It
holds random-number generation, bf16 rounding and the workload table only:
none of the loss or gradient arithmetic lives here, so sharing it does not
make the parity tests circular.
"""

from .generators import (  # noqa: F401
    IGNORE_INDEX,
    WORKLOADS,
    Workload,
    bf16_bits_to_f64,
    bf16_bits_to_f32,
    f64_to_bf16_bits,
    make_inputs,
    normal_bf16,
    splitmix64,
    uniform01,
    zipf_targets,
    apply_ignore,
    topk_targets,
    uniform_targets,
)
