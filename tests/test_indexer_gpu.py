"""GPU parity of the indexer top-k against the CPU indexer oracle.

The kernel accumulates scores in fp32 (bf16/fp16 products are exact in fp32), the
oracle in fp64: near-equal scores may order differently. So the comparison is by
score, per row, with tau = 1e-3 * (1 + max |I_ij|) (fp32 accumulation over H*d
terms stays orders of magnitude below): the count is min(k, visible keys), every
index is a distinct visible key, every selected key scores >= the oracle's k-th
score - tau, every visible key scoring > k-th + tau is selected, the returned
scores match the oracle's within tau and are non-increasing, and rows outside
the sequences keep their sentinel. Where every score of a row is exactly 0 (q = 0)
the tie order decides alone and the indices must equal the oracle's exactly.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.indexer as ix
from oracle.thd_attention import causal_shift
from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SENT = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


def run_indexer(batch: wl.IndexerBatch, kernel=bd.KERNEL_AUTO, max_seqlen_k=0, device="cuda"):
    q, k, w = batch.q.to(device), batch.k.to(device), batch.w.to(device)
    idx = torch.full((batch.cap_out, batch.topk), SENT, dtype=torch.int32, device=device)
    sc = torch.full((batch.cap_out, batch.topk), -123.0, dtype=torch.float32, device=device)
    ints = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    mask = torch.from_numpy(np.ascontiguousarray(batch.mask_type, dtype=np.int8)).to(device)
    qco = None if batch.q_causal_offset is None else ints(batch.q_causal_offset)
    plan = bd.indexer_plan_for_tensors(q, k, w, idx, batch.batch, batch.topk, max_seqlen_k, kernel)
    ws = bd.alloc_workspace(plan, device)
    bd.thd_indexer_topk(plan, q, k, w, idx, sc, ints(batch.cu_seqlens_q), ints(batch.cu_seqlens_kv),
                        ints(batch.off_q), ints(batch.off_k), ints(batch.off_out), mask, qco, ws)
    status = bd.thd_attn_read_status(plan, ws)
    torch.cuda.synchronize()
    return dict(idx=idx.cpu().numpy(), scores=sc.cpu().numpy(), status=status, plan=plan)


def _check_row(tag, row, srow, s_vis, ref_row, topk, exact=False):
    """One output row against the oracle's scores of the row's visible keys
    (``s_vis``, float64) and the oracle's selection ``ref_row``."""
    n_vis = s_vis.shape[0]
    n_out = min(topk, n_vis)
    assert (row[:n_out] >= 0).all() and (row[n_out:] == -1).all(), f"{tag}: count"
    sel = row[:n_out]
    assert len(set(sel.tolist())) == n_out and (sel < n_vis).all(), f"{tag}: bad index"
    assert np.isnan(srow[n_out:]).all()
    if n_out == 0:
        return
    tau = 1e-3 * (1.0 + float(np.abs(s_vis).max()))
    kth = float(s_vis[ref_row[n_out - 1]])
    assert (s_vis[sel] >= kth - tau).all(), f"{tag}: a selected key scores below the k-th"
    must = np.nonzero(s_vis > kth + tau)[0]
    assert set(must.tolist()) <= set(sel.tolist()), f"{tag}: a clearly better key is missing"
    assert np.abs(srow[:n_out] - s_vis[sel]).max() <= tau
    assert (np.diff(srow[:n_out]) <= 0).all(), f"{tag}: not in descending order"
    if exact:
        assert list(sel) == list(ref_row[:n_out]), f"{tag}: tie order"


def _n_visible(batch, b, i):
    lq, lk = int(batch.lens_q()[b]), int(batch.lens_k()[b])
    shift = causal_shift(int(batch.mask_type[b]), lq, lk,
                         None if batch.q_causal_offset is None else batch.q_causal_offset[b])
    return lk if shift is None else max(0, min(lk, i + shift + 1))


def _check_untouched(batch, res):
    written = np.zeros(batch.cap_out, dtype=bool)
    for b in range(batch.batch):
        written[int(batch.off_out[b]):int(batch.off_out[b]) + int(batch.lens_q()[b])] = True
    assert (res["idx"][~written] == SENT).all(), "an output row outside the sequences was written"
    assert (res["scores"][~written] == -123.0).all()


def check_indexer(batch: wl.IndexerBatch, res, exact_rows=False):
    init = np.full((batch.cap_out, batch.topk), SENT, dtype=np.int64)
    ref_idx, _, written = ix.indexer_topk(
        batch.q.to(torch.float64).numpy(), batch.k.to(torch.float64).numpy(), batch.w.to(torch.float64).numpy(),
        batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.off_q, batch.off_k, batch.off_out, batch.mask_type,
        batch.q_causal_offset, batch.topk, init)
    assert (res["idx"][~written] == SENT).all(), "an output row outside the sequences was written"
    assert (res["scores"][~written] == -123.0).all()
    lq, lk = batch.lens_q(), batch.lens_k()
    q64, k64, w64 = (t.to(torch.float64).numpy() for t in (batch.q, batch.k, batch.w))
    for b in range(batch.batch):
        if lq[b] == 0:
            continue
        qs, ks, os_ = int(batch.off_q[b]), int(batch.off_k[b]), int(batch.off_out[b])
        S = ix.indexer_scores_one(q64[qs:qs + lq[b]], k64[ks:ks + lk[b]], w64[qs:qs + lq[b]])
        for i in range(int(lq[b])):
            n_vis = _n_visible(batch, b, i)
            _check_row(f"seq {b} row {i}", res["idx"][os_ + i], res["scores"][os_ + i], S[i, :n_vis],
                       ref_idx[os_ + i], batch.topk, exact=exact_rows and not np.any(q64[qs + i]))


@pytest.mark.parametrize("kernel", [bd.KERNEL_AUTO, bd.KERNEL_SIMT])
@pytest.mark.parametrize("topk", [1, 16, 200])
def test_indexer_cp_chunks_small(topk, kernel):
    """Two documents, bottom-right causal query chunks at q_causal_offset = k_len - q_len."""
    batch = wl.indexer_cp(docs=2, k_len=1100, q_len=300, heads=8, d=64, topk=topk)
    res = run_indexer(batch, kernel=kernel)
    assert res["status"] == 0
    if kernel == bd.KERNEL_AUTO:
        assert res["plan"].kernel == bd.KERNEL_TCGEN05
    check_indexer(batch, res)


@pytest.mark.parametrize("heads,d", [(4, 64), (8, 128), (16, 64), (32, 128), (64, 128), (64, 64)])
def test_indexer_tc_shapes(heads, d):
    """Tensor-core scores for every supported head count (R = 128 / H query rows per
    MMA), ragged packs with gaps, mixed masks and ties."""
    batch = wl.indexer_random_pack(8400 + heads + d, batch=4, max_len=700, heads=heads, d=d, topk=64,
                                   dtype="bf16" if heads % 16 else "fp16", zero_q_rows=4)
    res = run_indexer(batch, kernel=bd.KERNEL_TCGEN05)
    assert res["status"] == 0
    check_indexer(batch, res, exact_rows=True)


@pytest.mark.parametrize("seed", range(8))
def test_indexer_random_packs(seed):
    rng = np.random.default_rng(8000 + seed)
    heads = [1, 4, 16, 64][seed % 4]
    d = [64, 128, 32, 16][(seed // 2) % 4]
    topk = [1, 7, 128, 300, 2048][seed % 5]
    batch = wl.indexer_random_pack(8100 + seed, batch=int(rng.integers(1, 6)), max_len=int(rng.integers(1, 700)),
                                   heads=heads, d=d, topk=topk, dtype=["bf16", "fp16"][seed % 2],
                                   zero_q_rows=5)
    res = run_indexer(batch)
    assert res["status"] == 0
    check_indexer(batch, res, exact_rows=True)


def test_indexer_long_rows_full_topk():
    """Rows of up to 3000 visible keys with k = 2048 (the radix-select path with a
    large k), plus rows with fewer visible keys than k."""
    batch = wl.indexer_random_pack(8200, batch=2, max_len=3000, heads=4, d=64, topk=2048, masks=(0, 2))
    res = run_indexer(batch)
    assert res["status"] == 0
    check_indexer(batch, res)


def test_indexer_key_length_over_bound_is_flagged():
    batch = wl.indexer_random_pack(8300, batch=3, max_len=200, heads=2, d=32, topk=8)
    lk = batch.lens_k()
    res = run_indexer(batch, max_seqlen_k=int(lk.max()) - 1)
    assert res["status"] & bd.DEV_BAD_LENGTH
    # the long sequence's rows are untouched
    b = int(np.argmax(lk))
    o, n = int(batch.off_out[b]), int(batch.lens_q()[b])
    assert (res["idx"][o:o + n] == SENT).all()


def test_indexer_128_heads_simt():
    """H = 128 (more heads than a tensor-core column group holds) runs on the SIMT
    scores with the same selection."""
    batch = wl.indexer_random_pack(8500, batch=3, max_len=400, heads=128, d=128, topk=32, zero_q_rows=2)
    res = run_indexer(batch)
    assert res["status"] == 0 and res["plan"].kernel == bd.KERNEL_SIMT
    check_indexer(batch, res, exact_rows=True)


def test_indexer_full_size_sampled():
    """The benchmark's workload in its launch configuration (two 65536-key
    documents, 4096-row chunks, H = 64, d = 128, k = 2048): sampled rows of both
    documents against the oracle, which scores each row on its own (rows are
    independent), and every row outside the sequences untouched."""
    batch = wl.indexer_cp()
    res = run_indexer(batch, max_seqlen_k=int(batch.lens_k().max()))
    assert res["status"] == 0 and res["plan"].kernel == bd.KERNEL_TCGEN05
    _check_untouched(batch, res)
    rng = np.random.default_rng(5)
    f64 = lambda t: t.to(torch.float64).numpy()
    for b in range(batch.batch):
        L, lk = int(batch.lens_q()[b]), int(batch.lens_k()[b])
        qs, ks, os_ = int(batch.off_q[b]), int(batch.off_k[b]), int(batch.off_out[b])
        kb = f64(batch.k[ks:ks + lk])
        rows = sorted({0, 1, 127, 128, 129, L - 2, L - 1, *rng.integers(0, L, size=4).tolist()})
        for i in rows:
            s_row = ix.indexer_scores_one(f64(batch.q[qs + i:qs + i + 1]), kb, f64(batch.w[qs + i:qs + i + 1]))
            n_vis = _n_visible(batch, b, i)
            vis = np.zeros((1, lk), dtype=bool)
            vis[0, :n_vis] = True
            ref_row = ix.select_topk(s_row, vis, batch.topk)[0]
            _check_row(f"doc {b} row {i}", res["idx"][os_ + i], res["scores"][os_ + i], s_row[0, :n_vis],
                       ref_row, batch.topk)


def test_indexer_zigzag_chunks_share_keys():
    """Zigzag context-parallel chunks of one 4096-token document (two ranks of
    cp_size 2, chunks of 1024 rows): four segments read overlapping key prefixes
    of the same key rows, 40 key units of 256 against 21 if key rows could not be
    shared -- the key-axis schedule must hold them all."""
    batch = wl.indexer_zigzag()
    assert int(np.sum(batch.lens_k())) > batch.k.shape[0]
    res = run_indexer(batch)
    assert res["status"] == 0 and res["plan"].kernel == bd.KERNEL_TCGEN05
    check_indexer(batch, res)
