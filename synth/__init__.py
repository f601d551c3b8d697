"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This package draws random numbers and lays them out; it holds none of the
attention arithmetic (no decode of E4M3, no dot products, no softmax).
"""
from .mla_inputs import (  # noqa: F401
    LATENT_DIM,
    ROPE_DIM,
    HEAD_DIM,
    PAGE_SIZE,
    SOFTMAX_SCALE,
    DecodeInputs,
    WORKLOADS,
    decode_inputs,
    kv_windows,
    merge_partials,
    page_selection,
    query_lens_ragged,
    ragged_lens,
    workload_inputs,
)
