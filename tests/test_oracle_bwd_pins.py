"""Pins of the backward oracle to facts outside itself (CPU only).

* central finite differences of the scalar brute-force forward (plain Python
  loops, ``oracle/brute.py``) on tiny ragged packs with every mask policy, causal
  offsets, windows, GQA and gaps between sequences;
* invariants of the softmax gradient: each row of dS sums to zero, so the keys'
  dK sum to zero per sequence and kv head; the keys' dV sum to the sum of dO over
  the live rows of the group;
* a special case with a closed form: a window of zero keys on a causal mask gives
  every live row exactly one key, so P = 1, dS = 0, dQ = dK = 0 and dV_j is the
  sum of dO over the rows that see key j;
* untouched rows outside the sequences;
* the context-parallel crop: a bottom-right chunk at q_causal_offset c has the
  gradients of full causal attention over its key prefix with dO = 0 on the
  other query rows;
* segments that share key rows (the zigzag chunks of one document, Megatron-LM
  PR #14): finite differences on a pack whose segments read the same K/V rows,
  and the zigzag chunks' summed dK / dV equal those of full causal attention
  over the document with dO = 0 outside the chunks.

``test_bwd_pins_catch_planted_mistakes`` plants plausible mistakes in the oracle
and checks that at least one pin fails for each.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle.backward as tb
from oracle.brute import brute_attention


def _tiny_pack(seed, h_q=2, h_kv=1, d=3, lens=((3, 4), (0, 2), (4, 4), (2, 5)), masks=(2, 0, 1, 2),
               qco=(1, 0, 0, -1), window=(-1, -1, 1, 2), gap=2):
    rng = np.random.default_rng(seed)
    lq = np.array([a for a, _ in lens])
    lk = np.array([b for _, b in lens])
    off_q = np.concatenate([[0], np.cumsum(lq + gap)])[:-1] + 1
    off_k = np.concatenate([[0], np.cumsum(lk + gap + 1)])[:-1]
    cap_q, cap_k = int(off_q[-1] + lq[-1] + gap), int(off_k[-1] + lk[-1] + gap)
    q = rng.standard_normal((cap_q, h_q, d))
    k = rng.standard_normal((cap_k, h_kv, d))
    v = rng.standard_normal((cap_k, h_kv, d))
    g = rng.standard_normal((cap_q, h_q, d))                 # dO, read at off_o = off_q
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    return dict(q=q, k=k, v=v, g=g, cu_q=cu_q, cu_k=cu_k, off_q=off_q, off_k=off_k,
                masks=np.array(masks), qco=np.array(qco), window=np.array(window))


def _oracle(p, scale=None):
    z = lambda a: np.full_like(a, 7.25)
    return tb.thd_attention_bwd(p["q"], p["k"], p["v"], p["g"], p["cu_q"], p["cu_k"], p["off_q"],
                                p["off_k"], p["off_k"], p["off_q"], p["masks"], p["qco"],
                                z(p["q"]), z(p["k"]), z(p["v"]), softmax_scale=scale,
                                window_left=p["window"])


def _brute_loss(p, q, k, v, scale):
    """L = sum over written O rows of <O, dO>, forward by scalar loops."""
    n_b = len(p["cu_q"]) - 1
    ql, kl, vl = q.tolist(), k.tolist(), v.tolist()
    o_init = np.zeros_like(q).tolist()
    st = [0.0] * (q.shape[0] * q.shape[1])
    o, _ = brute_attention(ql, kl, vl, list(p["cu_q"]), list(p["cu_k"]), list(p["off_q"]), list(p["off_k"]),
                           list(p["off_k"]), list(p["off_q"]), list(p["off_q"]), list(p["masks"]),
                           list(p["qco"]), o_init, st, q.shape[1], 1, scale=scale,
                           window_left=list(p["window"]))
    o = np.array(o)
    tot = 0.0
    for b in range(n_b):
        n = int(p["cu_q"][b + 1] - p["cu_q"][b])
        r = slice(int(p["off_q"][b]), int(p["off_q"][b]) + n)
        tot += float((o[r] * p["g"][r]).sum())
    return tot


def pin_finite_differences(seeds=(1, 2), make=_tiny_pack) -> float:
    """Max relative error of the oracle's gradients against central differences."""
    worst = 0.0
    for seed in seeds:
        p = make(seed)
        scale = 0.7
        dq, dk, dv, wq, wk, wv = _oracle(p, scale)
        eps = 1e-6
        for name, arr, grad, written in (("q", p["q"], dq, wq), ("k", p["k"], dk, wk), ("v", p["v"], dv, wv)):
            for idx in np.ndindex(arr.shape):
                if not written[idx[0]]:
                    continue
                plus, minus = arr.copy(), arr.copy()
                plus[idx] += eps
                minus[idx] -= eps
                args = {"q": p["q"], "k": p["k"], "v": p["v"]}
                args[name] = plus
                lp = _brute_loss(p, args["q"], args["k"], args["v"], scale)
                args[name] = minus
                lm = _brute_loss(p, args["q"], args["k"], args["v"], scale)
                fd = (lp - lm) / (2 * eps)
                err = abs(fd - grad[idx]) / max(1.0, abs(fd))
                worst = max(worst, err)
        assert worst < 1e-6, f"finite-difference mismatch {worst}"
    return worst


def pin_invariants(seed=5) -> float:
    p = _tiny_pack(seed, h_q=4, h_kv=2, d=5, lens=((6, 9), (5, 5), (7, 3)), masks=(0, 1, 2),
                   qco=(0, 0, 4), window=(-1, 3, 2))
    dq, dk, dv, *_ = _oracle(p)
    worst = 0.0
    group = p["q"].shape[1] // p["k"].shape[1]
    for b in range(len(p["cu_q"]) - 1):
        lq = int(p["cu_q"][b + 1] - p["cu_q"][b])
        lk = int(p["cu_k"][b + 1] - p["cu_k"][b])
        ks = slice(int(p["off_k"][b]), int(p["off_k"][b]) + lk)
        qs = int(p["off_q"][b])
        worst = max(worst, float(np.abs(dk[ks].sum(axis=0)).max(initial=0.0)))
        for g in range(p["k"].shape[1]):
            want = np.zeros(p["v"].shape[2])
            for h in range(g * group, (g + 1) * group):
                for i in range(lq):
                    # live row: at least one visible key
                    mt = int(p["masks"][b])
                    c = None if mt == 0 else (0 if mt == 1 else int(p["qco"][b]))
                    hi = lk if c is None else min(lk, i + c + 1)
                    w = int(p["window"][b])
                    lo = 0 if (c is None or w < 0) else max(0, i + c - w)
                    if hi > lo:
                        want += p["g"][qs + i, h]
            worst = max(worst, float(np.abs(dv[ks, g].sum(axis=0) - want).max(initial=0.0)))
    assert worst < 1e-9, f"invariant violated by {worst}"
    return worst


def pin_single_key_window(seed=6) -> float:
    """Window 0 on causal masks: one visible key per live row (closed form)."""
    p = _tiny_pack(seed, h_q=2, h_kv=1, d=4, lens=((5, 5), (4, 7)), masks=(1, 2), qco=(0, 2),
                   window=(0, 0))
    dq, dk, dv, wq, wk, wv = _oracle(p)
    worst = 0.0
    for b in range(2):
        lq = int(p["cu_q"][b + 1] - p["cu_q"][b])
        lk = int(p["cu_k"][b + 1] - p["cu_k"][b])
        c = 0 if p["masks"][b] == 1 else int(p["qco"][b])
        qs, ks = int(p["off_q"][b]), int(p["off_k"][b])
        worst = max(worst, float(np.abs(dq[qs:qs + lq]).max()), float(np.abs(dk[ks:ks + lk]).max()))
        want = np.zeros((lk, p["v"].shape[2]))
        for i in range(lq):
            j = i + c
            if 0 <= j < lk:
                want[j] += p["g"][qs + i].sum(axis=0)
        worst = max(worst, float(np.abs(dv[ks:ks + lk, 0] - want).max()))
    assert worst < 1e-12, f"single-key closed form off by {worst}"
    return worst


def pin_cp_crop(seed=8) -> float:
    """A context-parallel chunk (Megatron-LM PR #14): Lq query rows sitting at
    absolute rows c .. c + Lq - 1 of an Lk-key prefix, bottom-right with
    q_causal_offset = c, have the gradients of full causal self-attention over the
    Lk rows whose other query rows carry dO = 0 (they add nothing: dP = D = 0 there).
    dQ of the chunk = rows c .. c + Lq - 1 of the full dQ; dK and dV are equal."""
    rng = np.random.default_rng(seed)
    lk, c, lq, h, d = 11, 4, 5, 2, 3
    q_full = rng.standard_normal((lk, h, d))
    k, v = rng.standard_normal((lk, 1, d)), rng.standard_normal((lk, 1, d))
    g_full = np.zeros((lk, h, d))
    g_full[c:c + lq] = rng.standard_normal((lq, h, d))
    z = np.zeros
    full = tb.thd_attention_bwd(q_full, k, v, g_full, [0, lk], [0, lk], [0], [0], [0], [0], [1], None,
                                z(q_full.shape), z(k.shape), z(v.shape))
    chunk = tb.thd_attention_bwd(q_full[c:c + lq], k, v, g_full[c:c + lq], [0, lq], [0, lk], [0], [0], [0], [0],
                                 [2], [c], z((lq, h, d)), z(k.shape), z(v.shape))
    worst = max(float(np.abs(chunk[0] - full[0][c:c + lq]).max()), float(np.abs(chunk[1] - full[1]).max()),
                float(np.abs(chunk[2] - full[2]).max()))
    assert worst < 1e-12, f"CP chunk gradients differ from the full-prefix ones by {worst}"
    return worst


def _shared_key_pack(seed):
    """Three segments over one set of key rows (prefixes of it, each bottom-right
    at its own offset), a fourth with keys of its own, gaps between query rows."""
    rng = np.random.default_rng(seed)
    h_q, h_kv, d = 2, 1, 3
    lq = np.array([3, 2, 2, 3])
    lk = np.array([6, 4, 6, 4])
    off_q = np.array([1, 6, 10, 14])
    off_k = np.array([0, 0, 0, 8])
    cap_q, cap_k = 19, 13
    return dict(q=rng.standard_normal((cap_q, h_q, d)), k=rng.standard_normal((cap_k, h_kv, d)),
                v=rng.standard_normal((cap_k, h_kv, d)), g=rng.standard_normal((cap_q, h_q, d)),
                cu_q=np.concatenate([[0], np.cumsum(lq)]), cu_k=np.concatenate([[0], np.cumsum(lk)]),
                off_q=off_q, off_k=off_k, masks=np.array([2, 2, 0, 1]), qco=np.array([3, 2, 0, 0]),
                window=np.array([-1, 1, -1, -1]))


def pin_shared_keys_finite_differences(seed=9) -> float:
    """Central differences of the brute-force loss on a pack whose segments share
    K/V rows: a shared row's gradient is the sum over the segments reading it."""
    return pin_finite_differences(seeds=(seed,), make=_shared_key_pack)


def pin_zigzag_chunks(seed=10) -> float:
    """The zigzag query chunks of one document (chunks r and 2*cp-1-r of 2*cp equal
    chunks, cp = 2) as four segments over the SAME key rows, each bottom-right at its
    chunk start over the key prefix that ends with it: dQ of each chunk equals the
    full-document causal dQ of those rows, and the summed dK / dV equal the full
    ones when dO is zero on rows outside the chunks (here: none are outside)."""
    rng = np.random.default_rng(seed)
    doc, n_chunks, h, d = 16, 4, 2, 3
    c = doc // n_chunks
    q_full = rng.standard_normal((doc, h, d))
    k, v = rng.standard_normal((doc, 1, d)), rng.standard_normal((doc, 1, d))
    g_full = rng.standard_normal((doc, h, d))
    z = np.zeros
    full = tb.thd_attention_bwd(q_full, k, v, g_full, [0, doc], [0, doc], [0], [0], [0], [0], [1], None,
                                z(q_full.shape), z(k.shape), z(v.shape))
    order = [0, 3, 1, 2]                              # rank 0: chunks 0, 3; rank 1: chunks 1, 2
    q_seg = np.concatenate([q_full[x * c:(x + 1) * c] for x in order])
    g_seg = np.concatenate([g_full[x * c:(x + 1) * c] for x in order])
    cu_q = np.arange(0, len(order) * c + 1, c)
    lk = [(x + 1) * c for x in order]
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    seg = tb.thd_attention_bwd(q_seg, k, v, g_seg, cu_q, cu_k, cu_q[:-1], [0] * 4, [0] * 4, cu_q[:-1],
                               [2] * 4, [x * c for x in order], z(q_seg.shape), z(k.shape), z(v.shape))
    dq_want = np.concatenate([full[0][x * c:(x + 1) * c] for x in order])
    worst = max(float(np.abs(seg[0] - dq_want).max()), float(np.abs(seg[1] - full[1]).max()),
                float(np.abs(seg[2] - full[2]).max()))
    assert worst < 1e-12, f"zigzag chunk gradients differ from the full-document ones by {worst}"
    return worst


def pin_untouched_rows(seed=7) -> float:
    p = _tiny_pack(seed)
    dq, dk, dv, wq, wk, wv = _oracle(p)
    for arr, w in ((dq, wq), (dk, wk), (dv, wv)):
        assert (arr[~w] == 7.25).all(), "a row outside the sequences was written"
    # every sequence row is marked written
    for b in range(len(p["cu_q"]) - 1):
        lq = int(p["cu_q"][b + 1] - p["cu_q"][b])
        assert wq[int(p["off_q"][b]):int(p["off_q"][b]) + lq].all()
    return 0.0


PINS = {
    "finite_differences": pin_finite_differences,
    "invariants": pin_invariants,
    "single_key_window": pin_single_key_window,
    "untouched_rows": pin_untouched_rows,
    "cp_crop": pin_cp_crop,
    "shared_keys_finite_differences": pin_shared_keys_finite_differences,
    "zigzag_chunks": pin_zigzag_chunks,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_bwd_pin(name):
    PINS[name]()


# ----------------------------------------------------------- planted mistakes
def _variant(mistake):
    """The backward of one head with one plausible mistake planted."""
    def one(qb, kb, vb, dob, scale, shift, lower=None):
        len_q, len_k = qb.shape[0], kb.shape[0]
        if len_q == 0 or len_k == 0:
            return np.zeros_like(qb), np.zeros_like(kb), np.zeros_like(vb)
        s = scale * (qb @ kb.T)
        i_idx = np.arange(len_q)[:, None]
        j_idx = np.arange(len_k)[None, :]
        vis = np.ones_like(s, dtype=bool) if shift is None else (j_idx <= i_idx + shift)
        if lower is not None and mistake != "ignore_window":
            vis &= j_idx >= i_idx + lower
        s = np.where(vis, s, -np.inf)
        mx = s.max(axis=1)
        live = np.isfinite(mx)
        e = np.exp(s - np.where(live, mx, 0.0)[:, None])
        p_ = e / np.where(live, e.sum(axis=1), 1.0)[:, None]
        dp = dob @ vb.T
        if mistake == "drop_row_term":
            ds = p_ * dp
        elif mistake == "row_term_unweighted":
            ds = p_ * (dp - dp.mean(axis=1, keepdims=True))
        else:
            ds = p_ * (dp - (p_ * dp).sum(axis=1)[:, None])
        dv = (e.T @ dob) if mistake == "dv_unnormalised" else p_.T @ dob
        dq = (ds @ kb) * (1.0 if mistake == "no_scale_dq" else scale)
        dk = (ds.T @ qb) * scale
        if mistake == "dk_from_p":
            dk = (p_.T @ qb) * scale
        return dq, dk, dv
    one.__name__ = f"mutant_{mistake}"
    return one


@pytest.mark.parametrize("mistake", ["drop_row_term", "row_term_unweighted", "dv_unnormalised",
                                     "no_scale_dq", "ignore_window", "dk_from_p"])
def test_bwd_pins_catch_planted_mistakes(monkeypatch, mistake):
    monkeypatch.setattr(tb, "attention_one_head_bwd", _variant(mistake))
    failed = []
    for name, fn in PINS.items():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mistake}"


def test_shared_key_overwrite_mistake_is_caught(monkeypatch):
    """Writing each segment's dK / dV over the rows (the last segment wins) instead
    of summing the segments that share them."""
    orig = tb.thd_attention_bwd

    def overwrite(q, k, v, d_o, cu_q, cu_k, off_q, off_k, off_v, off_o, masks, qco, dq0, dk0, dv0, **kw):
        dq, dk, dv = np.array(dq0, dtype=float), np.array(dk0, dtype=float), np.array(dv0, dtype=float)
        wq, wk, wv = (np.zeros(len(x), dtype=bool) for x in (dq, dk, dv))
        win = kw.pop("window_left", None)
        for b in range(len(cu_q) - 1):
            lq, lk = int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])
            one = orig(q, k, v, d_o, [0, lq], [0, lk], [off_q[b]], [off_k[b]], [off_v[b]], [off_o[b]], [masks[b]],
                       None if qco is None else [qco[b]], dq, dk, dv,
                       window_left=None if win is None else [win[b]], **kw)
            dq, dk, dv = one[0], one[1], one[2]
            wq |= one[3]
            wk |= one[4]
            wv |= one[5]
        return dq, dk, dv, wq, wk, wv

    monkeypatch.setattr(tb, "thd_attention_bwd", overwrite)
    for pin in (pin_shared_keys_finite_differences, pin_zigzag_chunks):
        with pytest.raises(AssertionError):
            pin()


def test_gqa_head_map_mistake_is_caught(monkeypatch):
    """Summing dK/dV over interleaved instead of contiguous query-head groups."""
    orig = tb.thd_attention_bwd

    def interleaved(q, k, v, d_o, *a, **kw):
        h_q, h_kv = q.shape[1], k.shape[1]
        perm = np.array([(h % h_kv) * (h_q // h_kv) + h // h_kv for h in range(h_q)])
        dq, dk, dv, *w = orig(q[:, perm], k, v, d_o[:, perm], *a, **kw)
        inv = np.argsort(perm)
        return (dq[:, inv], dk, dv, *w)

    monkeypatch.setattr(tb, "thd_attention_bwd", interleaved)
    with pytest.raises(AssertionError):
        pin_invariants()
        pin_finite_differences()
