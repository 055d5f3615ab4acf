"""Oracle for the packed-THD sparse-attention indexer top-k -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may import this module.
The product path never calls it and shares no code with it.

The operation (Megatron-LM PR #14 "fix(dsa): align packed-CP indexer causal
masks": the indexer scores every key of a query's causal prefix, masked with the
same per-sequence policy and ``q_causal_offset`` as attention, and a top-k step
keeps the best keys per query row). The pages name the indexer but not its score
formula; this reading takes the published lightning-indexer score of
DeepSeek-V3.2's sparse attention, with ``H`` indexer heads per query row:

    I_ij = sum_h  w_ih * max(0, <q_ih, k_j>)

``q`` [rows, H, d] and ``k`` [rows, d] (one indexer key per token), ``w``
[rows, H] per-row head weights (any scale folded in; rows addressed like Q's). Visibility of key ``j``
for query row ``i`` is the attention forward's (mask 0 / 1 / 2 with
``q_causal_offset``). For each row, the selected keys are the ``topk`` visible
keys of largest ``I_ij``; with fewer visible keys all of them are selected. The
oracle lists them by descending score, equal scores by ascending key index,
then ``-1`` in the unused slots; indices are sequence-local key numbers
``0 .. len_k - 1``. Rows outside the sequences keep their prior contents.
"""
from __future__ import annotations

import numpy as np

from .thd_attention import causal_shift


def indexer_scores_one(qb: np.ndarray, kb: np.ndarray, wb: np.ndarray) -> np.ndarray:
    """I [len_q, len_k] in float64 for one sequence (no mask)."""
    dots = np.einsum("ihd,jd->ihj", qb, kb)                    # [len_q, H, len_k]
    return np.einsum("ih,ihj->ij", wb, np.maximum(dots, 0.0))


def select_topk(scores: np.ndarray, visible: np.ndarray, topk: int) -> np.ndarray:
    """Per row: visible keys ordered by (-score, key), first ``topk``, padded with -1."""
    n_rows = scores.shape[0]
    out = np.full((n_rows, topk), -1, dtype=np.int64)
    for i in range(n_rows):
        keys = np.nonzero(visible[i])[0]
        if keys.size == 0:
            continue
        order = np.lexsort((keys, -scores[i, keys]))             # primary: -score, then key
        chosen = keys[order[:topk]]
        out[i, :chosen.size] = chosen
    return out


def indexer_topk(q, k, w, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_out, mask_type,
                 q_causal_offset, topk, idx_init):
    """Top-k over one packed batch.

    ``q`` [cap_q, H, d], ``k`` [cap_k, d], ``w`` [cap_q, H] (the weights share Q's
    row offsets; any float dtype, upcast to float64 exactly), ``idx_init``
    [cap_out, topk] prior contents of the output.
    Returns ``(idx [cap_out, topk] int64, scores [cap_out, topk] float64 of the
    selected keys (NaN in unused slots), written [cap_out] bool)``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    idx = np.array(idx_init, dtype=np.int64, copy=True)
    sel = np.full(idx.shape, np.nan)
    written = np.zeros(idx.shape[0], dtype=bool)
    for b in range(len(cu_seqlens_q) - 1):
        len_q = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        len_k = int(cu_seqlens_kv[b + 1]) - int(cu_seqlens_kv[b])
        if len_q == 0:
            continue
        shift = causal_shift(int(mask_type[b]), len_q, len_k,
                             None if q_causal_offset is None else q_causal_offset[b])
        qs, ks, os_ = int(off_q[b]), int(off_k[b]), int(off_out[b])
        scores = indexer_scores_one(q[qs:qs + len_q], k[ks:ks + len_k], w[qs:qs + len_q])
        i_idx = np.arange(len_q)[:, None]
        j_idx = np.arange(len_k)[None, :]
        visible = np.ones((len_q, len_k), dtype=bool) if shift is None else (j_idx <= i_idx + shift)
        chosen = select_topk(scores, visible, topk)
        idx[os_:os_ + len_q] = chosen
        for i in range(len_q):
            m = chosen[i] >= 0
            sel[os_ + i, m] = scores[i, chosen[i][m]]
        written[os_:os_ + len_q] = True
    return idx, sel, written
