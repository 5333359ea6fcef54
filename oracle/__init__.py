"""fp64 CPU oracle for attention forward and backward.

TEST INFRASTRUCTURE: imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.
"""
from .ref import (  # noqa: F401
    attn_ref_probs,
    attn_ref_fwd,
    attn_ref_bwd,
    attn_ref_rows_fwd,
    attn_ref_rows_dq,
    attn_ref_keys_dkdv,
)
