"""GB300 (sm_103a) ring attention for context parallelism.

The compute path lives in ``libring_attn.so`` (hand-written tcgen05/TMA CUDA
kernels behind the C ABI in ``include/ring_attn.h``); this package is its
thin Python binding.
"""

from .ring_attn import (  # noqa: F401
    LAYOUTS,
    Plan,
    RingAttention,
    RingAttnError,
    dynamic_cp,
    load_library,
    ring_attn_bwd,
    ring_attn_fwd,
    ring_attention,
    workspace_status,
)
