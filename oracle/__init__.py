"""CPU oracle for packed-THD forward attention -- test infrastructure only.

Imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the library. Shares no code with the CUDA path.
"""
from .thd_attention import (MASK_CAUSAL_BOTTOM_RIGHT, MASK_CAUSAL_TOP_LEFT, MASK_NONE,
                            attention_one_head, causal_shift, thd_attention_fwd,
                            unmasked_entries, window_lower_shift)
from .brute import brute_attention
from .backward import attention_one_head_bwd, thd_attention_bwd
from .indexer import indexer_scores_one, indexer_topk, select_topk

__all__ = [
    "MASK_NONE", "MASK_CAUSAL_TOP_LEFT", "MASK_CAUSAL_BOTTOM_RIGHT", "attention_one_head",
    "causal_shift", "thd_attention_fwd", "unmasked_entries",
    "brute_attention", "window_lower_shift", "attention_one_head_bwd", "thd_attention_bwd",
    "indexer_scores_one", "indexer_topk", "select_topk",
]
