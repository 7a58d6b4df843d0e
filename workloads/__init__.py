"""Seeded synthetic inputs shared by the CUDA path's tests, the benchmark and the oracle's tests.

This package draws random numbers and arranges them into the shapes of the
few-shot, multi-turn and tree-of-thought workloads; it holds none of the
attention, radix-tree or quantisation arithmetic.
"""

from .generate import (  # noqa: F401
    Segment,
    Request,
    Workload,
    bf16_bits_to_f64,
    context_tokens,
    context_kv_bits,
    tiny_decode,
    fewshot_extend,
    batched_decode,
    multiturn_decode,
    tot_mixed,
    chunked_prefill,
    StreamRequest,
    ServingStream,
    serving_stream,
    token_kv,
    stream_query,
    generated_token,
    config,
    CONFIG_NAMES,
)
