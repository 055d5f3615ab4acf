"""GB300-native attention over packed, ragged THD batches: forward, backward
and the sparse-attention indexer top-k.

The compute path is the C-ABI library ``libthd_attn.so`` (CUDA kernels for
sm_103a); :mod:`.binding` marshals torch tensors into its calls. Importing this
package does not load the library; the first call does, and fails loudly when
the library has not been built.
"""
from .binding import (STATS_HEAD_MAJOR, STATS_TOKEN_MAJOR, KERNEL_AUTO, KERNEL_SIMT,
                      KERNEL_TCGEN05, ThdAttnError, ThdAttnPlan, library_path, load_library,
                      ThdAttention, thd_attention, thd_attn_backward, thd_attn_forward, thd_attn_fwd,
                      thd_attn_plan, thd_attn_read_status, thd_indexer)

__all__ = [
    "STATS_HEAD_MAJOR", "STATS_TOKEN_MAJOR", "KERNEL_AUTO", "KERNEL_SIMT", "KERNEL_TCGEN05",
    "ThdAttnError", "ThdAttnPlan", "library_path", "load_library", "thd_attn_forward",
    "thd_attn_fwd", "thd_attn_plan", "thd_attn_read_status", "thd_attn_backward", "thd_indexer",
    "ThdAttention", "thd_attention",
]
