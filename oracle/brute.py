"""Scalar brute-force oracle for packed-THD forward attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may use it. It restates the same definition as
``oracle/thd_attention.py`` with plain Python loops and ``math`` functions (no
numpy arithmetic), so the two agree only if both follow the definition:

* sequence ``b`` owns query rows ``off_q[b] .. off_q[b]+len_q-1`` and key/value
  rows ``off_k[b]`` / ``off_v[b]`` onward (per-tensor ragged offsets, cuDNN-frontend
  issue "THD lowering never reads the bound ragged offsets");
* row ``i`` sees key ``j < len_k`` when the mask is 0, ``j <= i`` when it is 1
  (top-left causal), ``j <= i + c`` when it is 2 (bottom-right causal, ``c`` the
  causal offset or ``len_k - len_q``), per TransformerEngine PR #3274 and
  Megatron-LM PR #14; with a left window ``w >= 0`` on a causal mask, also
  ``j >= i + c - w`` (``c = 0`` for mask 1);
* ``LSE_i`` is the natural log of the sum of ``exp`` of the scaled scores over the
  visible keys, ``O_i`` the probability-weighted sum of the visible values; a row
  with no visible key gets ``O_i = 0`` and ``LSE_i = -inf``.

Meant for tiny packs only (B <= a few, lengths <= ~16).
"""
from __future__ import annotations

import math


def brute_attention(q, k, v, cu_q, cu_k, off_q, off_k, off_v, off_o, off_s, masks, qco,
                    o_init, stats_init, stride_tok, stride_head, scale=None, window_left=None):
    """Same contract as ``thd_attention_fwd`` but on nested Python lists.

    q/k/v/o_init: nested lists [rows][heads][d] of floats; stats_init: flat list.
    Returns (o, stats) as nested/flat lists.
    """
    h_q = len(q[0]) if q else 0
    d = len(q[0][0]) if q else 0
    h_kv = len(k[0]) if k else 1
    group = h_q // h_kv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = [[list(col) for col in row] for row in o_init]
    stats = list(stats_init)
    for b in range(len(cu_q) - 1):
        lq = cu_q[b + 1] - cu_q[b]
        lk = cu_k[b + 1] - cu_k[b]
        for h in range(h_q):
            g = h // group
            for i in range(lq):
                qrow = q[off_q[b] + i][h]
                vis = []
                for j in range(lk):
                    if masks[b] == 0:
                        ok = True
                    else:
                        c = 0 if masks[b] == 1 else ((lk - lq) if qco is None else qco[b])
                        ok = j <= i + c
                        w = None if window_left is None else window_left[b]
                        if w is not None and w >= 0:
                            ok = ok and j >= i + c - w
                    if ok:
                        krow = k[off_k[b] + j][g]
                        acc = 0.0
                        for t in range(d):
                            acc += qrow[t] * krow[t]
                        vis.append((j, scale * acc))
                out_row = off_o[b] + i
                st_idx = (off_s[b] + i) * stride_tok + h * stride_head
                if not vis:
                    o[out_row][h] = [0.0] * len(v[0][0])
                    stats[st_idx] = -math.inf
                    continue
                mx = max(s for _, s in vis)
                tot = 0.0
                for _, s in vis:
                    tot += math.exp(s - mx)
                lse = mx + math.log(tot)
                acc_o = [0.0] * len(v[0][0])
                for j, s in vis:
                    p = math.exp(s - lse)
                    vrow = v[off_v[b] + j][g]
                    for t in range(len(acc_o)):
                        acc_o[t] += p * vrow[t]
                o[out_row][h] = acc_o
                stats[st_idx] = lse
    return o, stats
