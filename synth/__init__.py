"""Seeded synthetic inputs for the speculative-decoding verify step.

This package draws random numbers and lays them out in the shapes the verify
step consumes.  It holds none of the method's arithmetic (no softmax, no
acceptance test, no inverse-CDF, no attention): both the CPU oracle and the
CUDA library are fed from here, and nothing here is computed by either.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    workload,
    bf16_round,
    bf16_bits,
    bf16_from_bits,
    context_lengths,
    logits_inputs,
    kv_layout,
    kv_inputs_host,
    kv_inputs_device,
    random_tree,
)
