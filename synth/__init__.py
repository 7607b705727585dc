"""Seeded synthetic inputs for the dynamic-vocabulary draft LM head.

This package only draws random numbers and shapes them into the workloads the
method is run on (token streams, logits, LM-head weights, draft hidden
states).  It holds none of the method's arithmetic: no Top-K, no stream
update, no windowing, no gather and no projection.  Both the CPU oracle and
the CUDA path take their inputs from here; neither is imported by it.
"""

from .workloads import (  # noqa: F401
    CONFIGS,
    Workload,
    WorkloadConfig,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    get_config,
)
