"""Float64 CPU oracle for Mixture-of-Depths Attention (MoDA).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only users.  The GPU library never imports this package,
and this package imports nothing from the GPU library.
"""
from .oracle import (  # noqa: F401
    build,
    cores,
    forward,
    backward,
    backward_positions,
    backward_keys,
    decode,
    depth_store,
    depth_project,
    sliding_window,
    DTYPE_F64,
    DTYPE_F32,
    DTYPE_BF16,
)
