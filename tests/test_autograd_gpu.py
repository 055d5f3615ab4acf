"""The one-call Python API on the GPU: autograd through thd_attention (forward +
backward kernels) and the thd_indexer wrapper, against the CPU oracles."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import indexer_topk, thd_attention_bwd, thd_attention_fwd
from ragged_varlen_attention_gb300 import binding as bd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


def _packed(seed, lens, h_q, h_kv, d, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    t = int(sum(lens))
    q, k, v = (torch.randn((t, h, d), generator=g).to(dtype) for h in (h_q, h_kv, h_kv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, cu


@pytest.mark.parametrize("masks,window", [((2, 1, 0), None), ((1, 2, 2), (64, -1, 300))])
def test_autograd_matches_oracle(masks, window):
    lens = [300, 77, 513]
    h_q, h_kv, d = 4, 2, 128
    q, k, v, cu = _packed(21, lens, h_q, h_kv, d)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev).requires_grad_(True) for x in (q, k, v))
    cud = torch.from_numpy(cu).to(dev)
    mask = torch.tensor(masks, dtype=torch.int8, device=dev)
    win = None if window is None else torch.tensor(window, dtype=torch.int32, device=dev)
    o = bd.thd_attention(qd, kd, vd, cud, cud, mask_type=mask, window_left=win)
    g = torch.Generator().manual_seed(5)
    grad_o = torch.randn(o.shape, generator=g).to(torch.bfloat16)
    (o.float() * grad_o.to(dev).float()).sum().backward()
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    offs = cu[:-1]
    w_np = None if window is None else np.array(window)
    o_ref, _, _ = thd_attention_fwd(f64(q), f64(k), f64(v), cu, cu, offs, offs, offs, offs, offs, np.array(masks),
                                    None, np.zeros(tuple(o.shape)), np.zeros(q.shape[0] * h_q), h_q, 1,
                                    window_left=w_np)
    assert float(np.max(np.abs(f64(o) - o_ref))) <= 2e-2
    dq, dk, dv, *_ = thd_attention_bwd(f64(q), f64(k), f64(v), f64(grad_o), cu, cu, offs, offs, offs, offs,
                                       np.array(masks), None, np.zeros(tuple(q.shape)), np.zeros(tuple(k.shape)),
                                       np.zeros(tuple(v.shape)), window_left=w_np)
    for got, ref in ((qd.grad, dq), (kd.grad, dk), (vd.grad, dv)):
        err = float(np.max(np.abs(f64(got) - ref))) / max(1.0, float(np.max(np.abs(ref))))
        assert err <= 2e-2, err


def test_indexer_wrapper_matches_oracle():
    dev = torch.device("cuda", 0)
    lens_q, lens_k = [200, 150], [900, 400]
    g = torch.Generator().manual_seed(9)
    H, d, topk = 8, 64, 16
    qi = torch.randn((sum(lens_q), H, d), generator=g).to(torch.bfloat16)
    ki = torch.randn((sum(lens_k), d), generator=g).to(torch.bfloat16)
    w = torch.randn((sum(lens_q), H), generator=g)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    qco = np.array([lk - lq for lq, lk in zip(lens_q, lens_k)], dtype=np.int32)
    mask = torch.tensor([2, 2], dtype=torch.int8, device=dev)
    idx, sc = bd.thd_indexer(qi.to(dev), ki.to(dev), w.to(dev), torch.from_numpy(cu_q).to(dev),
                             torch.from_numpy(cu_k).to(dev), topk, mask_type=mask,
                             q_causal_offset=torch.from_numpy(qco).to(dev))
    f64 = lambda t: t.to(torch.float64).numpy()
    ref, ref_s, _ = indexer_topk(f64(qi), f64(ki), f64(w), cu_q, cu_k, cu_q[:-1], cu_k[:-1], cu_q[:-1], [2, 2], qco,
                                 topk, np.zeros((sum(lens_q), topk), dtype=np.int64))
    got_s = sc.cpu().numpy()
    # same selected scores up to the fp32 tolerance (sets may differ only among near-ties)
    tau = 1e-3 * (1.0 + np.nanmax(np.abs(ref_s)))
    assert np.nanmax(np.abs(got_s - ref_s)) <= tau
    assert (idx.cpu().numpy() >= 0).all()
