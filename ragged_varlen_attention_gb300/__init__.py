"""GB300-native forward attention over packed, ragged THD batches.

The compute path is the C-ABI library ``libthd_attn.so`` (CUDA kernels for
sm_103a); :mod:`.binding` marshals torch tensors into its calls. Importing this
package does not load the library; the first call does, and fails loudly when
the library has not been built.
"""
from .binding import (STATS_HEAD_MAJOR, STATS_TOKEN_MAJOR, KERNEL_AUTO, KERNEL_SIMT,
                      KERNEL_TCGEN05, ThdAttnError, ThdAttnPlan, library_path, load_library,
                      thd_attn_forward, thd_attn_fwd, thd_attn_plan, thd_attn_read_status)

__all__ = [
    "STATS_HEAD_MAJOR", "STATS_TOKEN_MAJOR", "KERNEL_AUTO", "KERNEL_SIMT", "KERNEL_TCGEN05",
    "ThdAttnError", "ThdAttnPlan", "library_path", "load_library", "thd_attn_forward",
    "thd_attn_fwd", "thd_attn_plan", "thd_attn_read_status",
]
