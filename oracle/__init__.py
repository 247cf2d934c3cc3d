"""CPU oracle for paged decode attention (fp64, plain loops).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use it; the library never does.  It shares no
code with the CUDA path; ``oracle.c`` states what it computes and where that is
defined.
"""
from .oracle import (  # noqa: F401
    F16, BF16, E4M3, build, lib, max_threads,
    f16_to_double, bf16_to_double, decode16, e4m3_to_double, float_to_e4m3,
    round_out, reshape_and_cache, decode, attend_range, copy_blocks, gather_blocks, scatter_blocks,
)
