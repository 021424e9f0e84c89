"""CPU oracle for the compressed sparse attention forward.

Test infrastructure only: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  The arithmetic lives in ``csa_oracle.c`` (plain C, double precision);
this package compiles it with gcc and wraps it with ctypes + numpy.
"""
from .oracle import (  # noqa: F401
    build,
    num_threads,
    set_num_threads,
    compressed_offsets,
    compress,
    compress_ex,
    indexer_logits,
    indexer_topk,
    attention,
    attention_bwd,
    indexer_kl,
    indexer_kl_bwd,
    quantize_fp8,
    dequantize_fp8,
    e4m3_value,
    KIND_CSA,
    KIND_HCA,
    KIND_WINDOW,
)
