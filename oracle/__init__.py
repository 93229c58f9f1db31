"""Float64 CPU oracle for the KDA decode recurrence and the fused KDA block.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg are the only callers.  The CUDA library never
imports, links or executes anything here, and nothing here imports the CUDA
library.
"""
from .oracle import (  # noqa: F401
    build,
    kda_decode,
    kda_block_tkg,
    BAD_SLOT,
    BAD_SEQLEN,
    GATE_SOFTPLUS,
    GATE_LOWER_BOUND,
    OUT_GATES,
)
