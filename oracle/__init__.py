"""fp64 CPU oracle for the decode-time KV-eviction pass.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the product path.  It shares
no code with the CUDA library.
"""
from .oracle import (  # noqa: F401
    AGE_SINCE_ACCESS,
    AGG_CUMULATIVE,
    AGG_EMA,
    AGE_SINCE_INSERT,
    REFRESH_FROZEN,
    REFRESH_FULL,
    REFRESH_LAZY,
    W_ENTROPY,
    W_VNORM,
    OracleParams,
    SequenceState,
    attention,
    build,
    ema,
    is_refresh,
    priority,
    select,
    set_threads,
    step,
)
