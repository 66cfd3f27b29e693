"""fp64 CPU oracle for paged GQA decode/verify attention, KV append, greedy
prefix acceptance, speculative sampling, greedy acceptance over a draft tree and the
cache compaction after it, and the one-byte (int8 / e4m3) KV cache.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's CPU
baseline leg may import this package; the product path never does.  It shares no
code with the CUDA library and does not import it.
"""
from .oracle import (  # noqa: F401
    build,
    f16_to_f64,
    bf16_to_f64,
    kv_append,
    kv_append_quant,
    quantize_row,
    quantize_cache,
    e4m3_to_f64,
    e4m3_from_float,
    attention,
    accept_prefix,
    accept_sampled,
    accept_tree,
    kv_compact,
    argmax,
    num_threads,
)
from .recompute import causal_attention_full  # noqa: F401
