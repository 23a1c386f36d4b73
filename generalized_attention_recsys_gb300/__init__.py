"""GB300-native Generalized Dot Product Attention (GDPA).

The compute runs in the CUDA library ``libgdpa.so`` (built from ``csrc/``);
this package only marshals arguments to its C-ABI. Importing the package does
not load the library; the first call does, and raises if it is missing.
"""

from ._lib import (ACTS, DTYPES, GdpaError, gdpa_bwd, gdpa_error_string, gdpa_fwd,  # noqa: F401
                   gdpa_get_status, gdpa_num_sms, gdpa_set_profile_events,
                   gdpa_workspace_bytes)
from .interface import flash_attn_func, flash_attn_varlen_func  # noqa: F401
