"""fp64 CPU oracle for the fused LM-head loss.

TEST INFRASTRUCTURE: only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library.
"""
from .oracle import (  # noqa: F401
    BF16, FP32, IGNORE_INDEX, REDUCE_SUM, REDUCE_TOKEN_MEAN,
    Problem, Result, Seam, active_mask, bf16_bits_to_f64, build, entropy, forward,
    forward_backward, grad_rows, gspo_seam, row_forward,
)
