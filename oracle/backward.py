"""Oracle for packed-THD attention BACKWARD -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` and the CPU-baseline leg of ``bench.py`` may import this module.
The product path never calls it and shares no code with it.

What it computes is the gradient of the forward pass defined in
``oracle/thd_attention.py`` (same addressing, masks, windows and GQA head map),
one sequence and one query head at a time, float64:

* Forward recalled: ``s_ij = scale <q_i, k_j>`` over visible keys,
  ``P_ij = exp(s_ij - LSE_i)``, ``O_i = sum_j P_ij v_j``.
* For an upstream gradient ``dO`` of the same shape as ``O`` (the loss is
  ``L = sum_i <O_i, dO_i>``), the chain rule through the softmax gives
    ``dV_j  = sum_i P_ij dO_i``
    ``dP_ij = <dO_i, v_j>``
    ``dS_ij = P_ij (dP_ij - sum_j' P_ij' dP_ij')``
    ``dQ_i  = scale sum_j dS_ij k_j``
    ``dK_j  = scale sum_i dS_ij q_i``
  with ``P_ij = 0`` on invisible keys. The row term ``sum_j' P_ij' dP_ij'``
  equals ``<dO_i, O_i>``, the form ragged SDPA backward engines compute from the
  saved O (cudnn-frontend PR #462 names the ``softmax_sum`` / ``dQ_accum``
  intermediates of that backward).
* GQA: ``dK`` and ``dV`` of key/value head ``g`` sum the contributions of every
  query head ``h`` with ``h // (h_q // h_kv) == g``.
* A dead row (no visible key) contributes nothing and gets ``dQ_i = 0``.
* Gradient tensors share their primal tensor's row offsets (``dQ`` at
  ``off_q``, ``dK`` at ``off_k``, ``dV`` at ``off_v``; ``dO`` is read at
  ``off_o``). Rows outside ``[off[b], off[b] + len[b])`` keep their prior values.
* Segments may share key rows: the zigzag query chunks of one document under
  context parallelism all attend to its key prefix (Megatron-LM PR #14, the
  packed-CP paths). The loss sums over every segment, so a K or V row read by
  several segments gets the SUM of their contributions (chain rule); a written
  row's prior content is replaced, never added to.

The saved forward Stats and O are not inputs here: the oracle recomputes P
from Q and K, so a kernel that reads Stats or O at the wrong place disagrees.
"""
from __future__ import annotations

import math

import numpy as np

from .thd_attention import causal_shift, window_lower_shift


def attention_one_head_bwd(qb: np.ndarray, kb: np.ndarray, vb: np.ndarray, dob: np.ndarray,
                           scale: float, shift: int | None, lower: int | None = None):
    """Gradients of one sequence and one query head, float64.

    ``qb`` [len_q, d], ``kb`` [len_k, d], ``vb`` [len_k, d_v], ``dob`` [len_q, d_v].
    Returns ``(dq [len_q, d], dk [len_k, d], dv [len_k, d_v])``.
    """
    len_q, len_k = qb.shape[0], kb.shape[0]
    dq = np.zeros_like(qb, dtype=np.float64)
    dk = np.zeros_like(kb, dtype=np.float64)
    dv = np.zeros_like(vb, dtype=np.float64)
    if len_q == 0 or len_k == 0:
        return dq, dk, dv
    s = scale * (qb @ kb.T)                                       # [len_q, len_k]
    i_idx = np.arange(len_q)[:, None]
    j_idx = np.arange(len_k)[None, :]
    visible = np.ones_like(s, dtype=bool) if shift is None else (j_idx <= i_idx + shift)
    if lower is not None:
        visible &= j_idx >= i_idx + lower
    s = np.where(visible, s, -np.inf)
    row_max = s.max(axis=1)
    live = np.isfinite(row_max)
    m = np.where(live, row_max, 0.0)
    e = np.exp(s - m[:, None])                                    # 0 on invisible keys
    tot = np.where(live, e.sum(axis=1), 1.0)
    p = e / tot[:, None]                                          # softmax rows; 0 rows when dead
    dv = p.T @ dob
    dp = dob @ vb.T
    row_term = (p * dp).sum(axis=1)
    ds = p * (dp - row_term[:, None])
    dq = scale * (ds @ kb)
    dk = scale * (ds.T @ qb)
    return dq, dk, dv


def thd_attention_bwd(q, k, v, d_o, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_v, off_o,
                      mask_type, q_causal_offset, dq_init, dk_init, dv_init, softmax_scale=None,
                      window_left=None):
    """Backward over one packed THD batch.

    q [cap_q, h_q, d], k [cap_k, h_kv, d], v [cap_v, h_kv, d], d_o [cap_o, h_q, d]:
    row views (any float dtype; upcast to float64 exactly). ``dq_init`` /
    ``dk_init`` / ``dv_init`` are the gradient buffers' prior contents (shapes of
    q / k / v); copies are returned with the sequences' rows written.

    Returns ``(dq, dk, dv, written_q, written_k, written_v)``; ``written_*`` mark
    the rows written in each buffer.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_o = np.asarray(d_o, dtype=np.float64)
    h_q, d = q.shape[1], q.shape[2]
    h_kv = k.shape[1]
    if h_q % h_kv != 0:
        raise ValueError("h_q must be a multiple of h_kv")
    group = h_q // h_kv
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    dq = np.array(dq_init, dtype=np.float64, copy=True)
    dk = np.array(dk_init, dtype=np.float64, copy=True)
    dv = np.array(dv_init, dtype=np.float64, copy=True)
    wq = np.zeros((dq.shape[0],), dtype=bool)
    wk = np.zeros((dk.shape[0],), dtype=bool)
    wv = np.zeros((dv.shape[0],), dtype=bool)
    # key and value gradients summed over every segment that reads a row
    sum_k = np.zeros_like(dk)
    sum_v = np.zeros_like(dv)
    for b in range(len(cu_seqlens_q) - 1):
        len_q = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        len_k = int(cu_seqlens_kv[b + 1]) - int(cu_seqlens_kv[b])
        shift = causal_shift(int(mask_type[b]), len_q, len_k,
                             None if q_causal_offset is None else q_causal_offset[b])
        lower = window_lower_shift(int(mask_type[b]), shift,
                                   None if window_left is None else window_left[b])
        qs, ks, vs, os_ = int(off_q[b]), int(off_k[b]), int(off_v[b]), int(off_o[b])
        acc_k = np.zeros((len_k, h_kv, d))
        acc_v = np.zeros((len_k, h_kv, v.shape[2]))
        for h in range(h_q):
            g = h // group
            gq, gk, gv = attention_one_head_bwd(q[qs:qs + len_q, h], k[ks:ks + len_k, g],
                                                v[vs:vs + len_k, g], d_o[os_:os_ + len_q, h],
                                                scale, shift, lower)
            dq[qs:qs + len_q, h] = gq
            acc_k[:, g] += gk
            acc_v[:, g] += gv
        sum_k[ks:ks + len_k] += acc_k
        sum_v[vs:vs + len_k] += acc_v
        wq[qs:qs + len_q] = True
        wk[ks:ks + len_k] = True
        wv[vs:vs + len_k] = True
    dk[wk] = sum_k[wk]
    dv[wv] = sum_v[wv]
    return dq, dk, dv, wq, wk, wv
