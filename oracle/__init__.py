"""Float64 CPU oracle for MLA speculative-verify decode.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The product library never
imports, links or runs anything here, and nothing here imports the product.
"""
from .oracle import (  # noqa: F401
    MODE_DIRECT,
    MODE_FOLDED,
    MODE_SPLIT,
    KV_BF16,
    KV_FP8_E4M3,
    build,
    decode,
    e4m3_to_double,
    fold_factor,
)
