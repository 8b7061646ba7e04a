"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle checks.

This package draws random tensors and nothing else: it holds none of the differential-attention
arithmetic (no scores, softmax, lambda, norm). Both sides of every parity check take their inputs
from here, so the oracle and the kernels see bit-identical values.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    bf16_round,
    make_decode_inputs,
    make_dout,
    make_gda_decode_inputs,
    make_gda_inputs,
    make_lambda_vectors,
    make_prefill_inputs,
    make_tiny_inputs,
    make_v2_decode_inputs,
    make_v2_inputs,
    page_cache,
    to_fp8_e4m3,
)
