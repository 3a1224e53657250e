"""GB300 (sm_103a) FlashAttention forward: a C-ABI library plus a thin binding.

``fa_fwd(q, k, v, scale=None, causal=False)`` computes exact softmax attention
on (batch, seq, heads, head_dim) tensors with GQA and a bottom-right causal
mask, returning O and the row log-sum-exp. All arithmetic runs in the
hand-written CUDA kernel of ``csrc/``; see ``include/fa.h`` for the ABI.
"""

from .api import (  # noqa: F401
    FAError,
    fa_debug_set_fault,
    fa_debug_set_schedule,
    fa_fwd,
    fa_fwd_strided,
    fa_fwd_host,
    fa_fwd_host_workspace_size,
    fa_merge,
    fa_fwd_decode,
    fa_decode_workspace_size,
    fa_status,
    fa_status_string,
    fa_version,
)

__version__ = "0.1.0"
