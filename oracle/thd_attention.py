"""Oracle for packed-THD forward attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module. The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

What it computes is the plain definition, one sequence and one query head at a
time, in float64 with the inputs upcast exactly from their storage type:

* Addressing (cuDNN-frontend issue "THD lowering never reads the bound ragged
  offsets", section "Concrete failure" and the per-tensor offsets proposal):
  sequence ``b`` has ``len_q = cu_seqlens_q[b+1] - cu_seqlens_q[b]`` query rows
  starting at physical row ``off_q[b]`` of Q; K, V, O and Stats each carry their
  own row offset (``off_k``, ``off_v``, ``off_o``, ``off_s``). Offsets are row
  units; rows outside ``[off[b], off[b] + len[b])`` are never read or written.
* Scores (scaled dot-product attention): ``s_ij = scale * <q_i, k_j>``.
* Visibility, per sequence (TransformerEngine PR #3274, the review comment that
  proposes ``attn_mask_type_per_seq``; Megatron-LM PR #14 "fix(dsa): align
  packed-CP indexer causal masks" for the causal offset):
    - 0 none:                 every key ``j < len_k``;
    - 1 top-left causal:      ``j <= i``  ("row i keeps keys j <= i");
    - 2 bottom-right causal:  ``j <= i + c`` with ``c = q_causal_offset[b]``
      (the key index of the chunk's local q[0]) or ``len_k - len_q`` when no
      offset tensor is given;
  always with ``j < len_k``. An optional per-sequence left window ``w`` bounds the
  causal masks from below (TransformerEngine PR #3274, "per-policy windows" /
  ``window_size_per_mask_type`` for bounded causal attention): with mask 1 or 2
  and ``w >= 0`` row ``i`` also needs ``j >= i + c - w`` (``c = 0`` for mask 1);
  ``w < 0`` or mask 0 leaves it unbounded.
* ``LSE_i = ln sum_{visible j} exp(s_ij)`` (natural log of the scaled scores,
  the FlashAttention / PyTorch-varlen ``softmax_lse`` convention referred to in
  cudnn-frontend PR #462, section "What");
  ``O_i = sum_j exp(s_ij - LSE_i) v_j``.
* A row with no visible key (the "dead-row path"): ``O_i = 0``, ``LSE_i = -inf``.
* Stats layouts (cudnn-frontend PR #462, "What" / "Root cause"): the LSE of
  (row ``r``, head ``h``) sits at flat index ``r * stride_tok + h * stride_head``
  -- token-major ``[t, h]`` is ``(h_q, 1)``, head-major ``[h, t]`` is ``(1, T_s)``.
* GQA: query head ``h`` reads key/value head ``h // (h_q // h_kv)``.

Every output element not listed above keeps the value it had on input.
"""
from __future__ import annotations

import math

import numpy as np

MASK_NONE = 0
MASK_CAUSAL_TOP_LEFT = 1
MASK_CAUSAL_BOTTOM_RIGHT = 2

# rows of one (sequence, head) block evaluated at once; bounds the S matrix held
# in memory at ROW_CHUNK x len_k float64 values
ROW_CHUNK = 256


def causal_shift(mask_type: int, len_q: int, len_k: int, q_causal_offset) -> int | None:
    """Key-index shift ``c`` such that row ``i`` sees keys ``j <= i + c``.

    ``None`` means no causal limit (mask type 0).
    """
    if mask_type == MASK_NONE:
        return None
    if mask_type == MASK_CAUSAL_TOP_LEFT:
        return 0
    if mask_type == MASK_CAUSAL_BOTTOM_RIGHT:
        if q_causal_offset is None:
            return len_k - len_q
        return int(q_causal_offset)
    raise ValueError(f"unknown mask type {mask_type}")


def window_lower_shift(mask_type: int, shift: int | None, window_left) -> int | None:
    """Row ``i`` additionally needs ``j >= i + lower``; None when unbounded."""
    if window_left is None or mask_type == MASK_NONE or int(window_left) < 0:
        return None
    return shift - int(window_left)


def attention_one_head(qb: np.ndarray, kb: np.ndarray, vb: np.ndarray, scale: float,
                       shift: int | None, rows: slice | None = None, lower: int | None = None):
    """O and LSE of one sequence and one query head, float64.

    ``qb`` [len_q, d], ``kb`` [len_k, d], ``vb`` [len_k, d_v]. ``rows``
    restricts the evaluation to a subset of query rows (rows are independent);
    ``lower`` is the window's lower shift (row i needs j >= i + lower).
    Returns ``(o [n, d_v], lse [n])``.
    """
    len_q, len_k = qb.shape[0], kb.shape[0]
    r0, r1 = (0, len_q) if rows is None else (rows.start, rows.stop)
    n = r1 - r0
    o = np.zeros((n, vb.shape[1]), dtype=np.float64)
    lse = np.full((n,), -np.inf, dtype=np.float64)
    if n == 0 or len_k == 0:
        return o, lse
    for c0 in range(r0, r1, ROW_CHUNK):
        c1 = min(r1, c0 + ROW_CHUNK)
        s = scale * (qb[c0:c1] @ kb.T)                       # [rows, len_k]
        i_idx = np.arange(c0, c1)[:, None]
        j_idx = np.arange(len_k)[None, :]
        visible = np.ones_like(s, dtype=bool) if shift is None else (j_idx <= i_idx + shift)
        if lower is not None:
            visible &= j_idx >= i_idx + lower
        s = np.where(visible, s, -np.inf)
        row_max = s.max(axis=1)
        live = np.isfinite(row_max)
        m = np.where(live, row_max, 0.0)
        e = np.exp(s - m[:, None])                           # exp(-inf) = 0 at masked keys
        total = e.sum(axis=1)
        with np.errstate(divide="ignore"):
            lse_c = np.where(live, m + np.log(np.where(live, total, 1.0)), -np.inf)
        o_c = np.where(live[:, None], (e @ vb) / np.where(live, total, 1.0)[:, None], 0.0)
        o[c0 - r0:c1 - r0] = o_c
        lse[c0 - r0:c1 - r0] = lse_c
    return o, lse


def thd_attention_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_v, off_o, off_s,
                      mask_type, q_causal_offset, o_init, stats_init, stats_stride_tok,
                      stats_stride_head, softmax_scale=None, row_subset=None, window_left=None):
    """Forward attention over one packed THD batch.

    q [cap_q, h_q, d], k [cap_k, h_kv, d], v [cap_v, h_kv, d]: logical row views
    of the inputs (any float dtype; upcast to float64 exactly).
    o_init [cap_o, h_q, d] and stats_init (flat) are the output buffers' prior
    contents; copies are returned with the attention rows written.
    ``q_causal_offset`` and ``window_left`` may be None. ``row_subset`` (optional) maps a sequence
    index to an iterable of query rows; only those rows are evaluated and
    written (rows are independent, so a subset is exact for those rows).

    Returns ``(o, stats, written)`` where ``written`` [cap_o] marks O rows
    written (Stats rows follow the same sequences via ``off_s``).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    h_q, d = q.shape[1], q.shape[2]
    h_kv = k.shape[1]
    if h_q % h_kv != 0:
        raise ValueError("h_q must be a multiple of h_kv")
    group = h_q // h_kv
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    o = np.array(o_init, dtype=np.float64, copy=True)
    stats = np.array(stats_init, dtype=np.float64, copy=True).reshape(-1)
    written = np.zeros((o.shape[0],), dtype=bool)
    n_seq = len(cu_seqlens_q) - 1
    for b in range(n_seq):
        len_q = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        len_k = int(cu_seqlens_kv[b + 1]) - int(cu_seqlens_kv[b])
        shift = causal_shift(int(mask_type[b]), len_q, len_k,
                             None if q_causal_offset is None else q_causal_offset[b])
        lower = window_lower_shift(int(mask_type[b]), shift,
                                   None if window_left is None else window_left[b])
        qs, ks, vs = int(off_q[b]), int(off_k[b]), int(off_v[b])
        os_, ss = int(off_o[b]), int(off_s[b])
        rows = None
        if row_subset is not None:
            sel = sorted(set(int(r) for r in row_subset.get(b, ())))
            rows = [r for r in sel if 0 <= r < len_q]
        for h in range(h_q):
            g = h // group
            qb = q[qs:qs + len_q, h, :]
            kb = k[ks:ks + len_k, g, :]
            vb = v[vs:vs + len_k, g, :]
            if rows is None:
                ob, lb = attention_one_head(qb, kb, vb, scale, shift, lower=lower)
                idx = np.arange(len_q)
            else:
                idx = np.array(rows, dtype=np.int64)
                ob = np.zeros((len(idx), v.shape[2]))
                lb = np.full((len(idx),), -np.inf)
                # runs of consecutive rows are evaluated together (rows are independent)
                starts = np.flatnonzero(np.diff(idx, prepend=-2) != 1)
                ends = np.append(starts[1:], len(idx))
                for a, e in zip(starts, ends):
                    ob[a:e], lb[a:e] = attention_one_head(qb, kb, vb, scale, shift,
                                                          rows=slice(int(idx[a]), int(idx[e - 1]) + 1),
                                                          lower=lower)
            o[os_ + idx, h, :] = ob
            stats[(ss + idx) * stats_stride_tok + h * stats_stride_head] = lb
        if rows is None:
            written[os_:os_ + len_q] = True
        else:
            written[os_ + np.array(rows, dtype=np.int64)] = True
    return o, stats, written


def unmasked_entries(cu_seqlens_q, cu_seqlens_kv, mask_type, q_causal_offset, h_q,
                     window_left=None) -> int:
    """Count of visible score entries summed over sequences and query heads."""
    total = 0
    for b in range(len(cu_seqlens_q) - 1):
        len_q = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        len_k = int(cu_seqlens_kv[b + 1]) - int(cu_seqlens_kv[b])
        shift = causal_shift(int(mask_type[b]), len_q, len_k,
                             None if q_causal_offset is None else q_causal_offset[b])
        lower = window_lower_shift(int(mask_type[b]), shift,
                                   None if window_left is None else window_left[b])
        if shift is None:
            total += len_q * len_k
            continue
        # row i sees keys [max(0, i + lower), min(len_k, i + shift + 1))
        i = np.arange(len_q, dtype=np.int64)
        hi = np.clip(i + shift + 1, 0, len_k)
        lo = np.zeros_like(i) if lower is None else np.clip(i + lower, 0, len_k)
        total += int(np.maximum(hi - lo, 0).sum())
    return total * h_q
