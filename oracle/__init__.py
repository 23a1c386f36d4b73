"""Float64 CPU oracle for GDPA (test infrastructure; never on the product path)."""

from .gdpa_ref import (  # noqa: F401
    ACTIVATIONS,
    LEAKY_SLOPE,
    act_fwd,
    act_grad,
    allowed_mask,
    gdpa_bwd,
    gdpa_fwd,
    unit_bwd,
    unit_fwd,
)
