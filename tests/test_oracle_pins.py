"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each pin is a function returning an error (0 for a pass) so that
``test_pins_catch_planted_mistakes`` can re-run it against oracles with a
deliberate mistake planted on the CPU and show that some pin fails.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import thd_attention as th
from oracle.brute import brute_attention
from ragged_varlen_attention_gb300 import workloads as wl
from tests.helpers import as_f64, max_abs_finite, oracle_on_batch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _run(q, k, v, cu_q, cu_k, off_q, off_k, off_v, off_o, off_s, masks, qco=None,
         o_init=None, st_init=None, stride_tok=None, stride_head=1, scale=None):
    h_q = q.shape[1]
    cap_o = int(np.max(np.asarray(off_o)[:-1] + np.diff(np.asarray(cu_q)))) if len(cu_q) > 1 else 0
    cap_o = max(cap_o, q.shape[0])
    if o_init is None:
        o_init = np.zeros((cap_o, h_q, v.shape[2]))
    if stride_tok is None:
        stride_tok = h_q
    if st_init is None:
        st_init = np.zeros(cap_o * h_q)
    return th.thd_attention_fwd(q, k, v, cu_q, cu_k, off_q, off_k, off_v, off_o, off_s, masks, qco,
                                o_init, st_init, stride_tok, stride_head, softmax_scale=scale)


def _shift(mask, lq, lk, qco_b):
    """Causal shift restated here (independent of the oracle's helper): row i sees
    keys j <= i + shift; None = no causal limit."""
    if mask == 0:
        return None
    if mask == 1:
        return 0
    return (lk - lq) if qco_b is None else int(qco_b)


def _n_visible(i, lk, shift):
    return lk if shift is None else max(0, min(lk, i + shift + 1))


def _dense_reference(qb, kb, vb, scale, mask_bool):
    """torch SDPA (fp64, CPU) and torch.logsumexp on one sequence/head: [L, d]."""
    qt = torch.from_numpy(qb)[None, None]
    kt = torch.from_numpy(kb)[None, None]
    vt = torch.from_numpy(vb)[None, None]
    m = torch.from_numpy(mask_bool)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)[0, 0]
    s = (qt @ kt.transpose(-1, -2))[0, 0] * scale
    s = s.masked_fill(~torch.from_numpy(mask_bool), float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


# ---------------------------------------------------------------- pins -----

def pin_identifier_layout() -> float:
    """Sequence 1 of [a a a 1 b b 2 2 c c c c 3] reads rows 4-5, not 3-4; identifier
    rows never influence any output; each sequence equals dense attention alone."""
    g = _golden("identifier_layout.json")
    cu = np.array(g["cu_seqlens"])
    padded = np.array(g["cu_seqlens_padded"])
    rng = np.random.default_rng(7)
    cap, h, d = len(g["tokens"]), 2, 8
    q, k, v = (rng.standard_normal((cap, h, d)) for _ in range(3))
    masks = np.array([1, 0, 1])
    o1, s1, written = _run(q, k, v, cu, cu, padded, padded, padded, padded, padded, masks)
    err = 0.0
    # identifier rows hold huge values in a second run: outputs must not move
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for r in g["identifier_rows"]:
        q2[r], k2[r], v2[r] = 1e6, -1e6, 1e6
    o2, s2, _ = _run(q2, k2, v2, cu, cu, padded, padded, padded, padded, padded, masks)
    err = max(err, float(np.max(np.abs(o1[written] - o2[written]))))
    err = max(err, float(np.max(np.abs(s1 - s2))))
    # written rows are exactly the sequence rows of the layout
    want = np.zeros(cap, dtype=bool)
    for rows in g["sequence_rows"]:
        want[rows] = True
    if not np.array_equal(written, want):
        return float("inf")
    if g["sequence_rows"][1][0] != padded[1] or g["prefix_of_lens_start_of_sequence_1"] != cu[1]:
        return float("inf")
    # per-sequence dense attention
    scale = 1 / math.sqrt(d)
    for b, rows in enumerate(g["sequence_rows"]):
        n = len(rows)
        mb = np.tril(np.ones((n, n), dtype=bool)) if masks[b] == 1 else np.ones((n, n), dtype=bool)
        for hh in range(h):
            od, ld = _dense_reference(q[rows, hh], k[rows, hh], v[rows, hh], scale, mb)
            err = max(err, float(np.max(np.abs(o1[rows, hh] - od))))
            err = max(err, float(np.max(np.abs(s1[np.array(rows) * h + hh] - ld))))
    return err


def pin_dense_special_case(seed=3) -> float:
    """Random pack: every sequence/head equals torch SDPA on that sequence alone."""
    bt = wl.random_pack(seed, batch=5, max_len=24, h_q=4, h_kv=2, d=16, dtype="fp32",
                        nan_pads=False, with_qco=True, stats_layout=0)
    o, st, _ = oracle_on_batch(bt)
    q, k, v = as_f64(bt.q), as_f64(bt.k), as_f64(bt.v)
    lq, lk = bt.lens_q(), bt.lens_k()
    scale = 1 / math.sqrt(bt.d)
    err = 0.0
    for b in range(bt.batch):
        if lq[b] == 0 or lk[b] == 0:
            continue
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                            None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        i = np.arange(lq[b])[:, None]
        j = np.arange(lk[b])[None, :]
        mb = np.ones((lq[b], lk[b]), dtype=bool) if c is None else (j <= i + c)
        live = mb.any(axis=1)
        for h in range(bt.h_q):
            g = h // (bt.h_q // bt.h_kv)
            qb = q[bt.off_q[b]:bt.off_q[b] + lq[b], h]
            kb = k[bt.off_k[b]:bt.off_k[b] + lk[b], g]
            vb = v[bt.off_v[b]:bt.off_v[b] + lk[b], g]
            od, ld = _dense_reference(qb, kb, vb, scale, mb)
            rows = bt.off_o[b] + np.arange(lq[b])
            err = max(err, float(np.max(np.abs(o[rows, h][live] - od[live]), initial=0)))
            srows = (bt.off_s[b] + np.arange(lq[b])) * bt.h_q + h
            err = max(err, float(np.max(np.abs(st[srows][live] - ld[live]), initial=0)))
            if not np.all(o[rows, h][~live] == 0) or not np.all(np.isneginf(st[srows][~live])):
                return float("inf")
    return err


def pin_torch_causal_flag(seed=4) -> float:
    """Top-left causal equals torch SDPA's own ``is_causal`` (square sequences)."""
    rng = np.random.default_rng(seed)
    L, h, d = 19, 2, 8
    q, k, v = (rng.standard_normal((L, h, d)) for _ in range(3))
    cu = np.array([0, L])
    o, st, _ = _run(q, k, v, cu, cu, cu, cu, cu, cu, cu, np.array([1]))
    err = 0.0
    for hh in range(h):
        qt, kt, vt = (torch.from_numpy(x[:, hh])[None, None] for x in (q, k, v))
        od = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[0, 0]
        err = max(err, float(np.max(np.abs(o[:, hh] - od.numpy()))))
    return err


def pin_cp_offset_crop(seed=5) -> float:
    """Bottom-right causal with offset c equals rows [c, c+Lq) of full causal attention
    over the Lk keys (query chunk placed at its absolute rows)."""
    rng = np.random.default_rng(seed)
    lk, lq, h, d = 40, 9, 2, 8
    err = 0.0
    for c in (0, 5, lk - lq, 17):
        k = rng.standard_normal((lk, h, d))
        v = rng.standard_normal((lk, h, d))
        qfull = rng.standard_normal((lk, h, d))
        qchunk = qfull[c:c + lq].copy()
        cu_full = np.array([0, lk])
        of, sf, _ = _run(qfull, k, v, cu_full, cu_full, cu_full, cu_full, cu_full, cu_full, cu_full,
                         np.array([1]))
        cu_q = np.array([0, lq])
        qco = np.array([c])
        oc, sc, _ = _run(qchunk, k, v, cu_q, cu_full, cu_q, cu_full, cu_full, cu_q, cu_q,
                         np.array([2]), qco=qco)
        err = max(err, float(np.max(np.abs(oc[:lq] - of[c:c + lq]))))
        err = max(err, float(np.max(np.abs(sc[:lq * h] - sf[c * h:(c + lq) * h]))))
        if c == lk - lq:  # the default offset (no tensor) is k_len - q_len
            od, sd, _ = _run(qchunk, k, v, cu_q, cu_full, cu_q, cu_full, cu_full, cu_q, cu_q,
                             np.array([2]))
            err = max(err, float(np.max(np.abs(od[:lq] - oc[:lq]))))
    return err


def pin_two_call_sum(seed=6) -> float:
    """Mixed per-sequence policy equals the sum of a causal call and a non-causal call,
    each treating the other policy's sequences as pads (pre-zeroed outputs)."""
    g = _golden("two_call_sum.json")
    toks = g["tokens"]
    rng = np.random.default_rng(seed)
    T, h, d = len(toks), 2, 8
    q, k, v = (rng.standard_normal((T, h, d)) for _ in range(3))

    def call(cu, padded, mask):
        cu, padded = np.array(cu), np.array(padded)
        masks = np.full(len(cu) - 1, mask)
        return _run(q, k, v, cu, cu, padded, padded, padded, padded, padded, masks,
                    o_init=np.zeros((T, h, d)), st_init=np.zeros(T * h))

    oa, sa, wa = call(g["causal_call"]["cu_seqlens"], g["causal_call"]["cu_seqlens_padded"], 1)
    ob, sb, wb = call(g["non_causal_call"]["cu_seqlens"], g["non_causal_call"]["cu_seqlens_padded"], 0)
    mixed = g["mixed_call_derived"]
    cu = np.array(mixed["cu_seqlens"])
    # the derived call must match the token string's runs
    runs = [0]
    for t in range(1, T):
        if toks[t] != toks[t - 1]:
            runs.append(t)
    runs.append(T)
    if list(cu) != runs:
        return float("inf")
    want_mask = [1 if toks[s].isdigit() else 0 for s in runs[:-1]]
    if want_mask != mixed["mask"]:
        return float("inf")
    om, sm, wm = _run(q, k, v, cu, cu, cu, cu, cu, cu, cu, np.array(mixed["mask"]),
                      o_init=np.zeros((T, h, d)), st_init=np.zeros(T * h))
    if np.any(wa & wb) or not np.array_equal(wa | wb, wm):
        return float("inf")
    err = float(np.max(np.abs(oa + ob - om)))
    st_rows = np.repeat(wa, h)
    lse_sum = np.where(st_rows, sa, sb)
    return max(err, float(np.max(np.abs(lse_sum - sm))))


def pin_closed_forms(seed=8) -> float:
    """V = 1 gives O = 1; Q = 0 gives LSE = ln(#visible) and O = mean of visible V;
    one-hot V gives the probability row (scipy softmax); GQA equals MHA with repeated
    K/V heads; head-major LSE is the transpose of token-major."""
    bt = wl.random_pack(seed, batch=4, max_len=12, h_q=4, h_kv=2, d=16, dtype="fp32",
                        nan_pads=False, with_qco=True, stats_layout=0)
    q, k, v = as_f64(bt.q), as_f64(bt.k), as_f64(bt.v)
    lq, lk = bt.lens_q(), bt.lens_k()
    st_tok, st_head = bt.stats_strides
    args = (bt.cu_seqlens_q, bt.cu_seqlens_kv, bt.off_q, bt.off_k, bt.off_v, bt.off_o, bt.off_s,
            bt.mask_type, bt.q_causal_offset)
    o0 = np.zeros((bt.cap_o, bt.h_q, bt.d))
    s0 = np.zeros(bt.stats_numel)
    err = 0.0
    # V == 1
    o, st, w = th.thd_attention_fwd(q, k, np.ones_like(v), *args, o0, s0, st_tok, st_head)
    for b in range(bt.batch):
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                            None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        for i in range(lq[b]):
            n = _n_visible(i, int(lk[b]), c)
            row = bt.off_o[b] + i
            want = 1.0 if n > 0 else 0.0
            err = max(err, float(np.max(np.abs(o[row] - want))))
    # Q == 0
    o, st, w = th.thd_attention_fwd(np.zeros_like(q), k, v, *args, o0, s0, st_tok, st_head)
    group = bt.h_q // bt.h_kv
    for b in range(bt.batch):
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                            None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        for i in range(lq[b]):
            n = _n_visible(i, int(lk[b]), c)
            for h in range(bt.h_q):
                lse = st[(bt.off_s[b] + i) * st_tok + h * st_head]
                if n == 0:
                    if not np.isneginf(lse):
                        return float("inf")
                    continue
                err = max(err, abs(lse - math.log(n)))
                mean_v = v[bt.off_v[b]:bt.off_v[b] + n, h // group].mean(axis=0)
                err = max(err, float(np.max(np.abs(o[bt.off_o[b] + i, h] - mean_v))))
    # one-hot V: V[j] = e_j (d >= len_k for this pack)
    dv = int(max(lk.max(), 1))
    onehot = np.zeros((v.shape[0], bt.h_kv, dv))
    for b in range(bt.batch):
        for j in range(lk[b]):
            onehot[bt.off_v[b] + j, :, j] = 1.0
    o, st, w = th.thd_attention_fwd(q, k, onehot, *args, np.zeros((bt.cap_o, bt.h_q, dv)), s0,
                                    st_tok, st_head)
    scale = 1 / math.sqrt(bt.d)
    for b in range(bt.batch):
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                            None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        for h in range(bt.h_q):
            kb = k[bt.off_k[b]:bt.off_k[b] + lk[b], h // group]
            for i in range(lq[b]):
                n = _n_visible(i, int(lk[b]), c)
                if n == 0:
                    continue
                s = scale * (kb[:n] @ q[bt.off_q[b] + i, h])
                p = scipy.special.softmax(s)
                err = max(err, float(np.max(np.abs(o[bt.off_o[b] + i, h, :n] - p))))
                err = max(err, float(np.max(np.abs(o[bt.off_o[b] + i, h, n:]), initial=0)))
    # GQA == MHA with repeated K/V heads
    o_g, s_g, _ = th.thd_attention_fwd(q, k, v, *args, o0, s0, st_tok, st_head)
    o_m, s_m, _ = th.thd_attention_fwd(q, np.repeat(k, group, axis=1), np.repeat(v, group, axis=1),
                                       *args, o0, s0, st_tok, st_head)
    err = max(err, float(np.max(np.abs(o_g - o_m))), max_abs_finite(s_g, s_m))
    # head-major == transpose of token-major
    _, s_h, _ = th.thd_attention_fwd(q, k, v, *args, o0, s0, 1, bt.cap_s)
    err = max(err, max_abs_finite(s_h.reshape(bt.h_q, bt.cap_s).T.reshape(-1), s_g))
    return err


def pin_dead_rows() -> float:
    """Rows with no visible key: O = 0 and LSE = -inf (zero-length K, negative shift)."""
    rng = np.random.default_rng(9)
    h, d = 2, 4
    q = rng.standard_normal((10, h, d))
    k = rng.standard_normal((10, h, d))
    v = rng.standard_normal((10, h, d))
    cu_q = np.array([0, 4, 10])
    cu_k = np.array([0, 0, 6])           # sequence 0 has no keys
    off = np.array([0, 4, 10])
    o, st, w = _run(q, k, v, cu_q, cu_k, off, off, off, off, off, np.array([0, 2]),
                    qco=np.array([0, -3]), o_init=np.full((10, h, d), 7.0))
    err = float(np.max(np.abs(o[0:4])))
    if not np.all(np.isneginf(st[0:4 * h])):
        return float("inf")
    # sequence 1: rows i with i - 3 < 0 are dead (i = 0, 1, 2); row 3 sees key 0 only
    err = max(err, float(np.max(np.abs(o[4:7]))))
    if not np.all(np.isneginf(st[4 * h:7 * h])):
        return float("inf")
    err = max(err, float(np.max(np.abs(o[7] - v[4]))))
    return err


def pin_brute_force(seeds=range(20, 30)) -> float:
    """Scalar-loop oracle agrees with the numpy oracle on tiny packs and the tiny
    padded workload."""
    batches = [wl.tiny_padded()] + [
        wl.random_pack(s, batch=3, max_len=7, h_q=2, h_kv=1 + (s % 2), d=4, dtype="fp32",
                       nan_pads=False) for s in seeds]
    err = 0.0
    for bt in batches:
        o, st, _ = oracle_on_batch(bt, o_init=torch.zeros(bt.cap_o, bt.h_q, bt.d),
                                   stats_init=torch.zeros(bt.stats_numel))
        st_tok, st_head = bt.stats_strides
        qco = None if bt.q_causal_offset is None else [int(x) for x in bt.q_causal_offset]
        ob, sb = brute_attention(as_f64(bt.q).tolist(), as_f64(bt.k).tolist(), as_f64(bt.v).tolist(),
                                 [int(x) for x in bt.cu_seqlens_q], [int(x) for x in bt.cu_seqlens_kv],
                                 [int(x) for x in bt.off_q], [int(x) for x in bt.off_k],
                                 [int(x) for x in bt.off_v], [int(x) for x in bt.off_o],
                                 [int(x) for x in bt.off_s], [int(x) for x in bt.mask_type], qco,
                                 np.zeros((bt.cap_o, bt.h_q, bt.d)).tolist(),
                                 [0.0] * bt.stats_numel, st_tok, st_head)
        err = max(err, float(np.max(np.abs(np.array(ob) - o))), max_abs_finite(np.array(sb), st))
    return err


def pin_window(seed=12) -> float:
    """Left windows on causal masks: a window at least as long as the sequence changes
    nothing; window 0 leaves exactly key i + c (O = v_{i+c}, LSE = its scaled score);
    mask 0 ignores the window; every sequence equals torch SDPA under the explicit
    band mask; the scalar loops agree."""
    err = 0.0
    bt = wl.random_pack(seed, batch=6, max_len=20, h_q=2, h_kv=1, d=8, dtype="fp32",
                        nan_pads=False, with_qco=True, stats_layout=0, with_window=True)
    q, k, v = as_f64(bt.q), as_f64(bt.k), as_f64(bt.v)
    lq, lk = bt.lens_q(), bt.lens_k()
    o0 = torch.zeros(bt.cap_o, bt.h_q, bt.d)
    s0 = torch.zeros(bt.stats_numel)
    # long windows == unbounded
    long_w = dict(bt.__dict__)
    long_w["window_left"] = np.full(bt.batch, 10 * 20, dtype=np.int32)
    a, sa, _ = oracle_on_batch(wl.ThdBatch(**long_w), o_init=o0, stats_init=s0)
    nw = dict(bt.__dict__)
    nw["window_left"] = None
    b_, sb, _ = oracle_on_batch(wl.ThdBatch(**nw), o_init=o0, stats_init=s0)
    err = max(err, float(np.max(np.abs(a - b_))), max_abs_finite(sa, sb))
    # window 0
    zw = dict(bt.__dict__)
    zw["window_left"] = np.zeros(bt.batch, dtype=np.int32)
    oz, sz, _ = oracle_on_batch(wl.ThdBatch(**zw), o_init=o0, stats_init=s0)
    scale = 1 / math.sqrt(bt.d)
    for b in range(bt.batch):
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                   None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        for i in range(lq[b]):
            for h in range(bt.h_q):
                row, srow = bt.off_o[b] + i, (bt.off_s[b] + i) * bt.h_q + h
                if c is None:                         # mask 0: unbounded, as without window
                    err = max(err, float(np.max(np.abs(oz[row, h] - b_[row, h]))))
                    continue
                j = i + c
                if 0 <= j < lk[b]:
                    err = max(err, float(np.max(np.abs(oz[row, h] - v[bt.off_v[b] + j, 0]))))
                    err = max(err, abs(sz[srow] - scale * float(q[bt.off_q[b] + i, h] @ k[bt.off_k[b] + j, 0])))
                elif not (np.all(oz[row, h] == 0) and np.isneginf(sz[srow])):
                    return float("inf")
    # torch SDPA under the explicit band mask, rows with a visible key
    o, st, _ = oracle_on_batch(bt, o_init=o0, stats_init=s0)
    for b in range(bt.batch):
        if lq[b] == 0 or lk[b] == 0:
            continue
        c = _shift(int(bt.mask_type[b]), int(lq[b]), int(lk[b]),
                   None if bt.q_causal_offset is None else bt.q_causal_offset[b])
        i = np.arange(lq[b])[:, None]
        j = np.arange(lk[b])[None, :]
        mb = np.ones((lq[b], lk[b]), dtype=bool) if c is None else (j <= i + c)
        w = int(bt.window_left[b])
        if c is not None and w >= 0:
            mb &= j >= i + c - w
        live = mb.any(axis=1)
        for h in range(bt.h_q):
            qb = q[bt.off_q[b]:bt.off_q[b] + lq[b], h]
            kb = k[bt.off_k[b]:bt.off_k[b] + lk[b], 0]
            vb = v[bt.off_v[b]:bt.off_v[b] + lk[b], 0]
            od, ld = _dense_reference(qb, kb, vb, scale, mb)
            rows = bt.off_o[b] + np.arange(lq[b])
            srows = (bt.off_s[b] + np.arange(lq[b])) * bt.h_q + h
            err = max(err, float(np.max(np.abs(o[rows, h][live] - od[live]), initial=0)))
            err = max(err, float(np.max(np.abs(st[srows][live] - ld[live]), initial=0)))
    # scalar loops
    tiny = wl.random_pack(seed + 1, batch=3, max_len=7, h_q=2, h_kv=1, d=4, dtype="fp32",
                          nan_pads=False, with_window=True)
    ot, stt, _ = oracle_on_batch(tiny, o_init=torch.zeros(tiny.cap_o, 2, 4), stats_init=torch.zeros(tiny.stats_numel))
    tok, head = tiny.stats_strides
    ob, sb2 = brute_attention(as_f64(tiny.q).tolist(), as_f64(tiny.k).tolist(), as_f64(tiny.v).tolist(),
                              [int(x) for x in tiny.cu_seqlens_q], [int(x) for x in tiny.cu_seqlens_kv],
                              [int(x) for x in tiny.off_q], [int(x) for x in tiny.off_k],
                              [int(x) for x in tiny.off_v], [int(x) for x in tiny.off_o],
                              [int(x) for x in tiny.off_s], [int(x) for x in tiny.mask_type],
                              None if tiny.q_causal_offset is None else [int(x) for x in tiny.q_causal_offset],
                              np.zeros((tiny.cap_o, 2, 4)).tolist(), [0.0] * tiny.stats_numel, tok, head,
                              window_left=[int(x) for x in tiny.window_left])
    err = max(err, float(np.max(np.abs(np.array(ob) - ot))), max_abs_finite(np.array(sb2), stt))
    return err


PINS = {
    "identifier_layout": (pin_identifier_layout, 1e-12),
    "dense_special_case": (pin_dense_special_case, 1e-12),
    "torch_causal_flag": (pin_torch_causal_flag, 1e-12),
    "cp_offset_crop": (pin_cp_offset_crop, 1e-12),
    "two_call_sum": (pin_two_call_sum, 1e-12),
    "closed_forms": (pin_closed_forms, 1e-12),
    "dead_rows": (pin_dead_rows, 0.0),
    "brute_force": (pin_brute_force, 1e-12),
    "window": (pin_window, 1e-12),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    fn, tol = PINS[name]
    err = fn()
    assert err <= tol, f"pin {name}: error {err}"


def test_stats_layout_example():
    """The page's head-major Stats strides (58880, 7360, 1, 1) are h_q x T_s with token
    stride 1 -- the layout the oracle's (stride_tok, stride_head) = (1, T_s) addresses."""
    g = _golden("stats_layout.json")
    h_q, t = g["h_q"], g["t_capacity"]
    seq_stride, head_stride, tok_stride, _ = g["head_major_stats_strides"]
    assert head_stride == t and tok_stride == 1 and seq_stride == h_q * t
    bt = wl.random_pack(11, batch=2, max_len=5, h_q=h_q, h_kv=h_q, d=4, dtype="fp32",
                        stats_layout=wl.STATS_HEAD_MAJOR, nan_pads=False)
    assert bt.stats_strides == (1, bt.cap_s)


def test_unmasked_entries_counts():
    """Visible-entry count of the cp_chunks shape: each of the 4096 rows of a chunk at
    offset 61440 sees 61441 + i keys."""
    cu_q = np.array([0, 4096, 8192])
    cu_k = np.array([0, 65536, 131072])
    n = oracle.unmasked_entries(cu_q, cu_k, np.array([2, 2]), np.array([61440, 61440]), 16)
    per_doc = sum(61441 + i for i in range(4096))
    assert n == 2 * 16 * per_doc == 8_321_564_672


# ------------------------------------------------- planted mistakes -----

def _mutant_shift_off_by_one(mask_type, len_q, len_k, qco):
    c = _ORIG_SHIFT(mask_type, len_q, len_k, qco)
    return None if c is None else c + 1


def _mutant_bottom_right_sign(mask_type, len_q, len_k, qco):
    c = _ORIG_SHIFT(mask_type, len_q, len_k, qco)
    if mask_type == 2:
        return len_q - len_k if qco is None else -int(qco)
    return c


_ORIG_SHIFT = th.causal_shift
_ORIG_ONE_HEAD = th.attention_one_head


def _mutant_no_scale(qb, kb, vb, scale, shift, rows=None):
    return _ORIG_ONE_HEAD(qb, kb, vb, 1.0, shift, rows)


def _mutant_swap_kv(qb, kb, vb, scale, shift, rows=None):
    if kb.shape == vb.shape:
        return _ORIG_ONE_HEAD(qb, vb, kb, scale, shift, rows)
    return _ORIG_ONE_HEAD(qb, kb, vb, scale, shift, rows)


def _mutant_dead_row_nan(qb, kb, vb, scale, shift, rows=None):
    o, lse = _ORIG_ONE_HEAD(qb, kb, vb, scale, shift, rows)
    lse = np.where(np.isneginf(lse), 0.0, lse)
    return o, lse


_ORIG_LOWER = th.window_lower_shift


def _mutant_window_off_by_one(mask_type, shift, window_left):
    lo = _ORIG_LOWER(mask_type, shift, window_left)
    return None if lo is None else lo + 1


_ORIG_FWD = th.thd_attention_fwd


def _mutant_offsets_from_prefix(q, k, v, cu_q, cu_k, off_q, off_k, off_v, off_o, off_s, *a, **kw):
    return _ORIG_FWD(q, k, v, cu_q, cu_k, cu_q, cu_k, cu_k, off_o, off_s, *a, **kw)


def _mutant_gqa_interleaved(q, k, v, *a, **kw):
    # maps query head h to kv head h % h_kv instead of h // group
    h_q, h_kv = q.shape[1], k.shape[1]
    if h_q == h_kv:
        return _ORIG_FWD(q, k, v, *a, **kw)
    idx = [(h % h_kv) * (h_q // h_kv) for h in range(h_q)]
    return _ORIG_FWD(q, np.repeat(k, h_q // h_kv, axis=1)[:, idx], np.repeat(v, h_q // h_kv, axis=1)[:, idx], *a, **kw)


@pytest.mark.parametrize("target,mutant", [
    ("causal_shift", _mutant_shift_off_by_one),
    ("causal_shift", _mutant_bottom_right_sign),
    ("attention_one_head", _mutant_no_scale),
    ("attention_one_head", _mutant_swap_kv),
    ("attention_one_head", _mutant_dead_row_nan),
    ("thd_attention_fwd", _mutant_offsets_from_prefix),
    ("thd_attention_fwd", _mutant_gqa_interleaved),
    ("window_lower_shift", _mutant_window_off_by_one),
])
def test_pins_catch_planted_mistakes(monkeypatch, target, mutant):
    """A mistake planted in the oracle (on the CPU) makes at least one pin fail."""
    monkeypatch.setattr(th, target, mutant)
    failed = []
    for name, (fn, tol) in PINS.items():
        if name == "brute_force" and target == "causal_shift":
            pass
        try:
            err = fn()
        except Exception:  # noqa: BLE001 - a crash also counts as a caught mistake
            err = float("inf")
        if not err <= tol:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutant.__name__}"


def test_row_subset_matches_brute_force_rows():
    """A row subset (single rows and runs of consecutive rows, in any order) gives
    the scalar brute force's values on exactly those rows and writes no other row."""
    batch = wl.random_pack(23, batch=3, max_len=40, h_q=2, h_kv=1, d=8, dtype="fp32", with_qco=True)
    lq = batch.lens_q()
    subset = {b: sorted({0, int(lq[b]) - 1, *range(3, 9), 11, 12, 20}) for b in range(batch.batch)}
    o_sub, s_sub, w_sub = oracle_on_batch(batch, row_subset=subset)
    st_tok, st_head = batch.stats_strides
    o_b, s_b = brute_attention(as_f64(batch.q).tolist(), as_f64(batch.k).tolist(), as_f64(batch.v).tolist(),
                               list(batch.cu_seqlens_q), list(batch.cu_seqlens_kv), list(batch.off_q),
                               list(batch.off_k), list(batch.off_v), list(batch.off_o), list(batch.off_s),
                               list(batch.mask_type), None if batch.q_causal_offset is None
                               else list(batch.q_causal_offset), as_f64(batch.o_init()).tolist(),
                               batch.stats_init().to(torch.float64).tolist(), st_tok, st_head)
    o_b, s_b = np.array(o_b), np.array(s_b)
    want = np.zeros(batch.cap_o, dtype=bool)
    for b in range(batch.batch):
        rows = [r for r in subset[b] if 0 <= r < lq[b]]
        want[batch.off_o[b] + np.array(rows, dtype=np.int64)] = True
        for h in range(batch.h_q):
            idx = (batch.off_s[b] + np.array(rows, dtype=np.int64)) * st_tok + h * st_head
            assert max_abs_finite(s_sub[idx], s_b[idx]) < 1e-12
    assert np.array_equal(w_sub, want)
    assert float(np.max(np.abs(o_sub[want] - o_b[want]), initial=0.0)) < 1e-12
    init = as_f64(batch.o_init())
    assert np.array_equal(o_sub[~want].view(np.uint64), init[~want].view(np.uint64))
