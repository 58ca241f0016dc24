"""fp64 CPU oracle for causal Polar Attention.

Test infrastructure: only the tests, the smoke check and the bench's
CPU-baseline leg may import this package.  The product path never does.
"""
from .polar_oracle import (  # noqa: F401
    DEFAULT_CONSTS,
    build_oracle,
    oracle_bwd,
    oracle_bwd_sampled,
    oracle_decode,
    oracle_decode_paged,
    oracle_fwd,
    oracle_memory_step,
    oracle_row_stats,
    oracle_rows,
)
