"""GB300-native selected-block (block-sparse) attention.

The compute path is libbsa.so (hand-written sm_103a CUDA behind a C ABI,
include/bsa.h); this package only builds it and marshals torch tensors into
its calls.
"""

from .api import (  # noqa: F401
    BLOCK_K_SUPPORTED,
    BLOCK_Q_SUPPORTED,
    BsaError,
    bsa_backward,
    bsa_backward_workspace_size,
    bsa_debug_wait_probe,
    bsa_device_status,
    bsa_forward,
    bsa_forward_causal,
    bsa_forward_workspace_size,
    bsa_get_last_error,
    bsa_select,
    bsa_select_noalloc,
    bsa_select_rope,
    bsa_select_workspace_size,
    bsa_validate_indices,
    bsa_version,
)
from .build import build  # noqa: F401
