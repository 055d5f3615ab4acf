"""Runs a ThdBatch through the C-ABI on the GPU and checks it against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl
from tests.helpers import max_abs_finite, oracle_on_batch

# O max-abs and LSE max-abs tolerances. bf16/fp16: the stated target. fp32: the
# SIMT kernel computes in fp32; score error ~ d * 2^-24 * |q||k| and exp/log
# approximations of a few ulp keep both well under 1e-4 for N(0,1) inputs.
TOL = {"bf16": (2e-2, 1e-3), "fp16": (2e-2, 1e-3), "fp32": (1e-4, 1e-4)}


def _strided(t: torch.Tensor, extra_heads: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """Device view of ``t`` [rows, h, d] whose token stride is (h + extra_heads) * d,
    e.g. one half of an interleaved [T, 2, H, D] buffer. Returns (view, backing)."""
    rows, h, d = t.shape
    backing = torch.empty((rows, h + extra_heads, d), dtype=t.dtype, device=device)
    backing.view(torch.uint8).fill_(0x5A)
    view = backing[:, :h, :]
    view.copy_(t.to(device))
    return view, backing


def run_thd(batch: wl.ThdBatch, kernel: int = bd.KERNEL_AUTO, device="cuda", gaps=(0, 0, 0, 0),
            stream=None, reps: int = 1, flags: int = 0, element_mult: int | None = None):
    """Launch the forward pass; returns host copies of O (view), Stats, O backing,
    the status word and the plan. With ``element_mult`` the offsets are passed in
    element units (row x token stride of each tensor, divided by the multiplier)."""
    q, qb = _strided(batch.q, gaps[0] * batch.h_q, device)
    k, kb = _strided(batch.k, gaps[1] * batch.h_kv, device)
    v, vb = _strided(batch.v, gaps[2] * batch.h_kv, device)
    o_host = batch.o_init()
    o, ob = _strided(o_host, gaps[3] * batch.h_q, device)
    ob.view(torch.uint8).fill_(wl.SENTINEL_BYTE)
    stats = batch.stats_init().to(device)
    ints = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    cu_q, cu_k = ints(batch.cu_seqlens_q), ints(batch.cu_seqlens_kv)
    row_offs = (batch.off_q, batch.off_k, batch.off_v, batch.off_o, batch.off_s)
    mult = 0
    if element_mult is not None:
        flags |= bd.FLAG_ELEMENT_OFFSETS
        mult = element_mult
        st_tok = batch.stats_strides[0]
        strides = (q.stride(0), k.stride(0), v.stride(0), o.stride(0), st_tok)
        div = max(1, element_mult)
        conv = []
        for off, sd in zip(row_offs, strides):
            e = off.astype(np.int64) * sd
            assert (e % div == 0).all()
            conv.append(e // div)
        row_offs = conv
    offs = [ints(x) for x in row_offs]
    mask = torch.from_numpy(np.ascontiguousarray(batch.mask_type, dtype=np.int8)).to(device)
    qco = None if batch.q_causal_offset is None else ints(batch.q_causal_offset)
    win = None if batch.window_left is None else ints(batch.window_left)
    plan = bd.plan_for_tensors(q, k, v, o, batch.batch, batch.cap_s, batch.stats_layout,
                               batch.softmax_scale, kernel, flags, mult)
    ws = bd.alloc_workspace(plan, device)
    for _ in range(reps):
        if win is None:
            bd.thd_attn_fwd(plan, q, k, v, o, stats, cu_q, cu_k, *offs, mask, qco, ws, stream)
        else:
            bd.thd_attn_fwd_window(plan, q, k, v, o, stats, cu_q, cu_k, *offs, mask, qco, win, ws,
                                   stream)
    status = bd.thd_attn_read_status(plan, ws, stream)
    torch.cuda.synchronize()
    return dict(o=o.cpu(), o_backing=ob.cpu(), stats=stats.cpu(), status=status, plan=plan,
                ws=ws, dev=dict(q=q, k=k, v=v, o=o, stats=stats, cu_q=cu_q, cu_k=cu_k, offs=offs,
                                mask=mask, qco=qco, win=win))


def check_parity(batch: wl.ThdBatch, res, row_subset=None, tol=None):
    """Element-wise comparison with the oracle on written rows, bitwise sentinel
    check everywhere else. Returns (o_err, lse_err)."""
    tol_o, tol_l = TOL[batch.dtype] if tol is None else tol
    o_ref, s_ref, written = oracle_on_batch(batch, row_subset=row_subset)
    o_gpu = res["o"].to(torch.float64).numpy()
    s_gpu = res["stats"].to(torch.float64).numpy()
    # rows the oracle wrote
    o_err = float(np.max(np.abs(o_gpu[written] - o_ref[written]), initial=0.0))
    assert np.isfinite(o_gpu[written]).all(), "non-finite O in a written row"
    st_tok, st_head = batch.stats_strides
    lq = batch.lens_q()
    s_idx = []
    for b in range(batch.batch):
        rows = np.arange(lq[b]) if row_subset is None else np.array(sorted(row_subset.get(b, [])),
                                                                     dtype=np.int64)
        rows = rows[rows < lq[b]]
        for h in range(batch.h_q):
            s_idx.append((batch.off_s[b] + rows) * st_tok + h * st_head)
    s_idx = np.concatenate(s_idx) if s_idx else np.zeros(0, dtype=np.int64)
    lse_err = max_abs_finite(s_gpu[s_idx], s_ref[s_idx])
    assert o_err <= tol_o, f"O max-abs {o_err} > {tol_o}"
    assert lse_err <= tol_l, f"LSE max-abs {lse_err} > {tol_l}"
    return o_err, lse_err


def check_untouched(batch: wl.ThdBatch, res):
    """Every O/Stats byte outside the sequences' rows still holds the sentinel."""
    lq = batch.lens_q()
    ob = res["o_backing"].view(torch.uint8).numpy().reshape(batch.cap_o, -1)
    h, d = batch.h_q, batch.d
    elem = res["o"].element_size()
    written = np.zeros(batch.cap_o, dtype=bool)
    for b in range(batch.batch):
        written[batch.off_o[b]:batch.off_o[b] + lq[b]] = True
    # pad rows: every byte; written rows: the bytes past the h*d elements (token gap)
    assert (ob[~written] == wl.SENTINEL_BYTE).all(), "a pad row of O was written"
    assert (ob[written][:, h * d * elem:] == wl.SENTINEL_BYTE).all(), "O token gap was written"
    st = res["stats"].view(torch.uint8).numpy().reshape(-1, 4)
    from tests.helpers import written_stats_mask
    wm = written_stats_mask(batch)
    assert (st[~wm] == wl.SENTINEL_BYTE).all(), "a pad element of Stats was written"
