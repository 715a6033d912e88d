"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package holds shapes and random-number draws only: no step of the decoder's
arithmetic lives here, so neither side can borrow the other's math through it.
"""
from .shapes import SHAPES, Shape, Workload, WORKLOADS
from .inputs import (
    tensor_names,
    tensor_shapes,
    param_count,
    make_weights,
    make_prompt,
    make_batch_prompts,
    round_to_bf16,
    bf16_bits,
)

__all__ = [
    "SHAPES", "Shape", "Workload", "WORKLOADS", "tensor_names", "tensor_shapes",
    "param_count", "make_weights", "make_prompt", "make_batch_prompts",
    "round_to_bf16", "bf16_bits",
]
