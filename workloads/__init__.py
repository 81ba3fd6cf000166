"""Seeded synthetic decode workloads for the NVFP4-compressed MLA cache.

This package only draws random inputs (block tables, top-k index sets,
bf16 latent/rope/query values). It holds none of the method's arithmetic:
no quantisation, no dequantisation, no attention. Both the CUDA path and
the CPU oracle take their inputs from here.
"""
from .gen import (  # noqa: F401
    CONFIG_NAMES,
    Workload,
    make_workload,
    make_queries,
    make_rows,
    make_append_batch,
    referenced_tokens,
    all_tokens,
    redraw_indices,
    bf16_from_f32,
    f32_from_bf16,
)
