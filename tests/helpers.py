"""Shared test helpers: run the oracle on a ThdBatch and compare results."""
from __future__ import annotations

import numpy as np
import torch

from oracle import thd_attention as _th


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def oracle_on_batch(batch, o_init=None, stats_init=None, row_subset=None):
    """Oracle result for ``batch`` with the sentinel-filled buffers as prior content."""
    o0 = batch.o_init() if o_init is None else o_init
    s0 = batch.stats_init() if stats_init is None else stats_init
    st_tok, st_head = batch.stats_strides
    return _th.thd_attention_fwd(
        as_f64(batch.q), as_f64(batch.k), as_f64(batch.v),
        batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.off_q, batch.off_k, batch.off_v,
        batch.off_o, batch.off_s, batch.mask_type, batch.q_causal_offset,
        as_f64(o0), s0.to(torch.float64).numpy(), st_tok, st_head,
        softmax_scale=batch.softmax_scale, row_subset=row_subset,
        window_left=getattr(batch, "window_left", None))


def written_stats_mask(batch) -> np.ndarray:
    """Flat boolean mask of Stats elements the attention must write."""
    st_tok, st_head = batch.stats_strides
    m = np.zeros(batch.stats_numel, dtype=bool)
    lq = batch.lens_q()
    for b in range(batch.batch):
        rows = np.arange(int(batch.off_s[b]), int(batch.off_s[b]) + int(lq[b]))
        for h in range(batch.h_q):
            m[rows * st_tok + h * st_head] = True
    return m


def max_abs_finite(a: np.ndarray, b: np.ndarray) -> float:
    """Max |a-b| where -inf must match -inf exactly (returns inf otherwise)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    ninf_a, ninf_b = np.isneginf(a), np.isneginf(b)
    if not np.array_equal(ninf_a, ninf_b):
        return float("inf")
    if np.isnan(a).any() or np.isnan(b).any():
        return float("inf")
    fin = ~ninf_a
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(a[fin] - b[fin])))
