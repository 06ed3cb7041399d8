"""CPU fp64 oracle for the block-quantised decode GEMV (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it.  See ``qmv_oracle.c`` for the definition
and its citations.
"""
from .oracle import (  # noqa: F401
    FMT_Q4_0,
    FMT_Q8_0,
    FMT_Q2W,
    block_bytes,
    build,
    dequant_row,
    half_to_double,
    max_threads,
    moe,
    qmv,
    qmv_rows,
    swiglu,
)
