"""Float64 CPU oracle for rational-softmax attention.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the product package.
"""
from .ra_oracle import (  # noqa: F401
    POWER,
    SUPPORT,
    default_scale,
    ra_attention_bwd,
    ra_attention_fwd,
    ra_attention_head_bwd,
    ra_attention_head_fwd,
    ra_attention_rows_fwd,
    ra_phi,
    ra_softmax,
    ra_softmax_bwd,
)
from .ra_module import layer_norm, ra_attention_module_bwd, ra_attention_module_fwd  # noqa: F401
from .ra_tiled import ra_attention_tiled_head  # noqa: F401
