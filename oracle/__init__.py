"""fp64 CPU oracle for the attention forward/backward (test infrastructure).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this package.  The CUDA library never calls it and has no CPU fallback.
Every function is pinned by tests that do not reuse its own code: central finite
differences, library routines (scaled_dot_product_attention + autograd in fp64,
logsumexp), closed forms, identities and brute-force masks.
"""
from .attention import (  # noqa: F401
    causal_mask, full_mask, head_forward, head_backward, dense_forward, dense_backward,
    thd_backward, sparse_token, sparse_forward, sparse_backward, sparse_dkv_rows,
    sparse_valid,
)
