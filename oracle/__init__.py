"""CPU oracle for exact softmax attention (test infrastructure only).

Plain, slow, float64 NumPy restatement of what the attention path computes.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
it; the product path (the CUDA library and its binding) never does, and the two
share no code. See attention.py for the definitions and the passages they
follow.
"""

from .attention import (  # noqa: F401
    attention_forward,
    attention_forward_rows,
    attention_backward,
    attention_fwd_bwd_rows,
    attention_probabilities,
    tiled_forward,
    tiled_backward,
    softmax_rows,
)
