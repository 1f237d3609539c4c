"""Seeded synthetic inputs for the decode-time KV-eviction pass.

This package only draws random tensors and rounds them to bf16; it holds none
of the eviction method's arithmetic.  Both the CUDA path (through the Python
binding) and the CPU oracle take their inputs from here, so that the two sides
see bit-identical bf16 values.
"""
from .gen import (  # noqa: F401
    Geometry,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    rope_table,
    tiny_workload,
    llama8b_workload,
    needle_blocks,
    paged_workload,
    memdecay_workload,
    region_labels,
    region_spans,
    REGION_NAMES,
    REGION_HALF_LIVES,
    REGION_PINNED,
    DECODE_REGION,
)
