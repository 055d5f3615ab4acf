"""Pins of the indexer top-k oracle to facts outside itself (CPU only).

* brute force: scores by scalar loops and selection by Python's ``sorted`` with
  the same (descending score, ascending key) order, on tiny ragged packs with
  every mask policy and causal offsets;
* a special case that reduces to a library routine: one head, weight 1 and
  positive vectors make the score a plain dot product, whose top-k for an
  unmasked row is ``numpy.argsort`` of the negated dot products (stable);
* the properties the pages measure: zero causally-out-of-bounds indices and the
  number of selected keys equal to min(k, visible keys); for a context-parallel
  chunk the bottom-right mask with q_causal_offset gives row i the prefix
  0 .. i + c, while the top-left mask gives the chunk-local window 0 .. i
  (Megatron-LM PR #14);
* selected scores dominate every unselected visible score;
* the zigzag context-parallel chunks of one document select what the
  full-document causal indexer selects for the same rows (the pages' exact
  index-parity check).

``test_indexer_pins_catch_planted_mistakes`` plants mistakes in the oracle and
checks that a pin fails for each.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle.indexer as ix


def _pack(seed, H=3, d=4, lens=((4, 6), (0, 3), (5, 5), (3, 9)), masks=(2, 0, 1, 2), qco=(2, 0, 0, 7),
          gap=2, topk=4):
    rng = np.random.default_rng(seed)
    lq = np.array([a for a, _ in lens])
    lk = np.array([b for _, b in lens])
    off_q = np.concatenate([[0], np.cumsum(lq + gap)])[:-1] + 1
    off_k = np.concatenate([[0], np.cumsum(lk + gap + 1)])[:-1]
    off_o = np.concatenate([[0], np.cumsum(lq + 1)])[:-1] + 2
    cap_q, cap_k = int(off_q[-1] + lq[-1] + gap), int(off_k[-1] + lk[-1] + gap)
    cap_o = int(off_o[-1] + lq[-1] + 1)
    return dict(q=rng.standard_normal((cap_q, H, d)), k=rng.standard_normal((cap_k, d)),
                w=rng.standard_normal((cap_q, H)), cu_q=np.concatenate([[0], np.cumsum(lq)]),
                cu_k=np.concatenate([[0], np.cumsum(lk)]), off_q=off_q, off_k=off_k, off_o=off_o,
                masks=np.array(masks), qco=np.array(qco), topk=topk, cap_o=cap_o)


def _run(p, qco=True):
    init = np.full((p["cap_o"], p["topk"]), -7, dtype=np.int64)
    return ix.indexer_topk(p["q"], p["k"], p["w"], p["cu_q"], p["cu_k"], p["off_q"], p["off_k"], p["off_o"],
                           p["masks"], p["qco"] if qco else None, p["topk"], init)


def _visible(mask, i, j, lq, lk, c):
    if j >= lk:
        return False
    if mask == 0:
        return True
    if mask == 1:
        return j <= i
    return j <= i + c


def pin_brute_force(seeds=(1, 2, 3)) -> float:
    for seed in seeds:
        p = _pack(seed)
        idx, sel, written = _run(p)
        H, d = p["q"].shape[1], p["q"].shape[2]
        for b in range(len(p["cu_q"]) - 1):
            lq = int(p["cu_q"][b + 1] - p["cu_q"][b])
            lk = int(p["cu_k"][b + 1] - p["cu_k"][b])
            for i in range(lq):
                cand = []
                for j in range(lk):
                    if not _visible(int(p["masks"][b]), i, j, lq, lk, int(p["qco"][b])):
                        continue
                    s = 0.0
                    for h in range(H):
                        dot = 0.0
                        for e in range(d):
                            dot += p["q"][p["off_q"][b] + i, h, e] * p["k"][p["off_k"][b] + j, e]
                        s += p["w"][p["off_q"][b] + i, h] * max(0.0, dot)
                    cand.append((-s, j))
                want = [j for _, j in sorted(cand)[:p["topk"]]]
                want += [-1] * (p["topk"] - len(want))
                got = list(idx[p["off_o"][b] + i])
                assert got == want, f"seq {b} row {i}: {got} != {want}"
    return 0.0


def pin_dot_product_special_case(seed=4) -> float:
    rng = np.random.default_rng(seed)
    lq, lk, d, topk = 6, 40, 8, 7
    q = np.abs(rng.standard_normal((lq, 1, d)))
    k = np.abs(rng.standard_normal((lk, d)))
    w = np.ones((lq, 1))
    idx, _, _ = ix.indexer_topk(q, k, w, [0, lq], [0, lk], [0], [0], [0], [0], None, topk,
                                np.zeros((lq, topk), dtype=np.int64))
    dots = q[:, 0, :] @ k.T
    for i in range(lq):
        want = np.argsort(-dots[i], kind="stable")[:topk]
        assert list(idx[i]) == list(want), f"row {i}"
    return 0.0


def pin_causal_bounds_and_counts(seed=5) -> float:
    """CP chunk: 8 query rows at the end of a 40-key prefix (c = 32)."""
    rng = np.random.default_rng(seed)
    lq, lk, H, d, topk = 8, 40, 2, 4, 16
    q, k, w = rng.standard_normal((lq, H, d)), rng.standard_normal((lk, d)), rng.standard_normal((lq, H))
    init = np.zeros((lq, topk), dtype=np.int64)
    br, _, _ = ix.indexer_topk(q, k, w, [0, lq], [0, lk], [0], [0], [0], [2], [lk - lq], topk, init)
    tl, _, _ = ix.indexer_topk(q, k, w, [0, lq], [0, lk], [0], [0], [0], [1], None, topk, init)
    for i in range(lq):
        for got, limit in ((br[i], i + lk - lq), (tl[i], i)):
            chosen = got[got >= 0]
            assert chosen.size == min(topk, limit + 1), f"row {i}: {chosen.size} keys"
            assert (chosen <= limit).all(), f"row {i}: causally out-of-bounds index"
            assert len(set(chosen.tolist())) == chosen.size
            assert (got[chosen.size:] == -1).all()
    return 0.0


def pin_dominance(seed=6) -> float:
    p = _pack(seed, H=2, d=6, lens=((7, 30), (5, 12)), masks=(2, 0), qco=(20, 0), topk=5)
    idx, sel, _ = _run(p)
    for b in range(2):
        lq = int(p["cu_q"][b + 1] - p["cu_q"][b])
        lk = int(p["cu_k"][b + 1] - p["cu_k"][b])
        qs, ks = int(p["off_q"][b]), int(p["off_k"][b])
        scores = ix.indexer_scores_one(p["q"][qs:qs + lq], p["k"][ks:ks + lk], p["w"][qs:qs + lq])
        for i in range(lq):
            got = idx[p["off_o"][b] + i]
            chosen = set(got[got >= 0].tolist())
            vis = [j for j in range(lk) if _visible(int(p["masks"][b]), i, j, lq, lk, int(p["qco"][b]))]
            rest = [scores[i, j] for j in vis if j not in chosen]
            if rest and chosen:
                assert min(scores[i, j] for j in chosen) >= max(rest)
            s = [scores[i, j] for j in got[got >= 0]]
            assert all(x >= y for x, y in zip(s, s[1:])), "not in descending score order"
    return 0.0


def pin_zigzag_chunks_equal_full_document(seed=8) -> float:
    """The pages' check of packed context-parallel chunks (Megatron-LM PR #14): the
    zigzag chunks of one document (cp_size 2: rank r holds chunks r and 3 - r of 12
    rows), each a segment over the key prefix that ends with it, bottom-right aligned
    at q_causal_offset = its first global row, select exactly what the full-document
    causal indexer selects for the same rows (overlap 1, nothing causally out of
    bounds). The chunk-local top-left mask selects differently for the later chunks."""
    rng = np.random.default_rng(seed)
    n, c, H, d, topk = 48, 12, 2, 5, 6
    q, k, w = rng.standard_normal((n, H, d)), rng.standard_normal((n, d)), rng.standard_normal((n, H))
    full, _, _ = ix.indexer_topk(q, k, w, [0, n], [0, n], [0], [0], [0], [1], None, topk,
                                 np.zeros((n, topk), dtype=np.int64))
    chunks = [0, 3, 1, 2]                                       # rank 0, then rank 1
    cu_q = np.concatenate([[0], np.cumsum([c] * 4)])
    cu_k = np.concatenate([[0], np.cumsum([(ch + 1) * c for ch in chunks])])
    starts = [ch * c for ch in chunks]
    for masks, qco in (([2] * 4, starts), ([1] * 4, None)):
        got, _, _ = ix.indexer_topk(q, k, w, cu_q, cu_k, starts, [0] * 4, starts, masks, qco, topk,
                                    np.zeros((n, topk), dtype=np.int64))
        if qco is not None:
            assert (got == full).all(), "zigzag chunks disagree with the full document"
            for ch in chunks:
                rows = got[ch * c:(ch + 1) * c]
                assert (rows < (np.arange(ch * c, (ch + 1) * c) + 1)[:, None]).all()
        else:
            assert (got[:c] == full[:c]).all()                  # chunk 0: local == global
            assert not (got == full).all(), "a chunk-local mask should select differently"
    return 0.0


def pin_untouched_rows(seed=7) -> float:
    p = _pack(seed)
    idx, _, written = _run(p)
    assert (idx[~written] == -7).all()
    return 0.0


PINS = {"brute_force": pin_brute_force, "dot_product_special_case": pin_dot_product_special_case,
        "causal_bounds_and_counts": pin_causal_bounds_and_counts, "dominance": pin_dominance,
        "untouched_rows": pin_untouched_rows, "zigzag_chunks": pin_zigzag_chunks_equal_full_document}


@pytest.mark.parametrize("name", sorted(PINS))
def test_indexer_pin(name):
    PINS[name]()


_orig_scores = ix.indexer_scores_one
_orig_select = ix.select_topk


def _no_relu(qb, kb, wb):
    return np.einsum("ih,ihj->ij", wb, np.einsum("ihd,jd->ihj", qb, kb))


def _weights_of_next_row(qb, kb, wb):
    return _orig_scores(qb, kb, np.roll(wb, 1, axis=0))


def _smallest_first(scores, visible, topk):
    return _orig_select(-scores, visible, topk)


def _ties_by_larger_key(scores, visible, topk):
    out = np.full((scores.shape[0], topk), -1, dtype=np.int64)
    for i in range(scores.shape[0]):
        keys = np.nonzero(visible[i])[0][::-1]
        order = np.argsort(-scores[i, keys], kind="stable")
        chosen = keys[order[:topk]]
        out[i, :chosen.size] = chosen
    return out


def _causal_off_by_one(scores, visible, topk):
    v = visible.copy()
    v[:, 1:] |= visible[:, :-1]
    return _orig_select(scores, v, topk)


@pytest.mark.parametrize("target,mutant", [
    ("indexer_scores_one", _no_relu),
    ("indexer_scores_one", _weights_of_next_row),
    ("select_topk", _smallest_first),
    ("select_topk", _ties_by_larger_key),
    ("select_topk", _causal_off_by_one),
])
def test_indexer_pins_catch_planted_mistakes(monkeypatch, target, mutant):
    monkeypatch.setattr(ix, target, mutant)
    failed = []
    for name, fn in PINS.items():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    assert failed, f"no pin caught {mutant.__name__}"
