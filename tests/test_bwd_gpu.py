"""GPU parity of the backward pass (dQ, dK, dV) against the CPU backward oracle.

Inputs: the forward's O and Stats come from the forward ORACLE (cast to the
storage types), dO is seeded N(0, 1) with NaN in pad rows, and every gradient
buffer starts as a byte sentinel so untouched rows are checked bit for bit.

Tolerance (normalised max error, |gpu - ref|_inf / max(1, |ref|_inf) per
gradient): bf16/fp16 2e-2 -- the gradients are stored in a 16-bit type (2^-9 /
2^-11 relative) and D_i = <dO_i, O_i> is formed from a 16-bit O, which shifts dS
by P_ij * |dO_i| * |O_i| * 2^-9 at most; fp32 1e-4 (fp32 arithmetic throughout).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle.backward as ob
from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl
from tests.gpu_harness import _strided
from tests.helpers import as_f64, oracle_on_batch

pytestmark = pytest.mark.gpu

KERNELS = [bd.KERNEL_AUTO, bd.KERNEL_SIMT]
TOL = {"bf16": 2e-2, "fp16": 2e-2, "fp32": 1e-4}
SENTINEL = wl.SENTINEL_BYTE


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


def _dout(batch: wl.ThdBatch, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    t = torch.randn((batch.cap_o, batch.h_q, batch.d), generator=g, dtype=torch.float32)
    lq = batch.lens_q()
    keep = np.zeros(batch.cap_o, dtype=bool)
    for b in range(batch.batch):
        keep[batch.off_o[b]:batch.off_o[b] + lq[b]] = True
    t[torch.from_numpy(~keep)] = float("nan")
    return t.to(batch.torch_dtype)


def run_bwd(batch: wl.ThdBatch, kernel=bd.KERNEL_AUTO, gaps=(0,) * 8, seed=0, flags=0, device="cuda",
            device_mask=None, element_mult=None):
    """Forward outputs from the oracle, then the backward through the C ABI
    (``device_mask`` replaces the mask array passed to the device; with
    ``element_mult`` the offsets go in element units: row x token stride of the
    primal tensor, divided by the multiplier)."""
    o_ref, s_ref, written = oracle_on_batch(batch)
    o_host = batch.o_init().clone()
    o_host[torch.from_numpy(written)] = torch.from_numpy(o_ref[written]).to(batch.torch_dtype)
    stats_host = torch.from_numpy(s_ref.astype(np.float32))
    d_o_host = _dout(batch, seed)
    q, _ = _strided(batch.q, gaps[0] * batch.h_q, device)
    k, _ = _strided(batch.k, gaps[1] * batch.h_kv, device)
    v, _ = _strided(batch.v, gaps[2] * batch.h_kv, device)
    o, _ = _strided(o_host, gaps[3] * batch.h_q, device)
    d_o, _ = _strided(d_o_host, gaps[4] * batch.h_q, device)
    grads = []
    for src, gap, h in ((batch.q, gaps[5], batch.h_q), (batch.k, gaps[6], batch.h_kv), (batch.v, gaps[7], batch.h_kv)):
        view, backing = _strided(torch.zeros_like(src), gap * h, device)
        backing.view(torch.uint8).fill_(SENTINEL)
        grads.append((view, backing))
    (dq, dqb), (dk, dkb), (dv, dvb) = grads
    stats = stats_host.to(device)
    ints = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    row_offs = (batch.off_q, batch.off_k, batch.off_v, batch.off_o, batch.off_s)
    mult = 0
    if element_mult is not None:
        flags |= bd.FLAG_ELEMENT_OFFSETS
        mult = element_mult
        strides = (q.stride(0), k.stride(0), v.stride(0), o.stride(0), batch.stats_strides[0])
        conv = []
        for off, sd in zip(row_offs, strides):
            e = off.astype(np.int64) * sd
            assert (e % max(1, mult) == 0).all()
            conv.append(e // max(1, mult))
        row_offs = conv
    offs = [ints(x) for x in row_offs]
    mask = torch.from_numpy(np.ascontiguousarray(batch.mask_type if device_mask is None else device_mask,
                                                 dtype=np.int8)).to(device)
    qco = None if batch.q_causal_offset is None else ints(batch.q_causal_offset)
    win = None if batch.window_left is None else ints(batch.window_left)
    plan = bd.plan_bwd_for_tensors(q, k, v, o, d_o, dq, dk, dv, batch.batch, batch.cap_s, batch.stats_layout,
                                   batch.softmax_scale, kernel, flags, mult)
    ws = bd.alloc_workspace(plan, device)
    bd.thd_attn_bwd(plan, q, k, v, o, d_o, stats, dq, dk, dv, ints(batch.cu_seqlens_q),
                    ints(batch.cu_seqlens_kv), *offs, mask, qco, win, ws)
    status = bd.thd_attn_read_status(plan, ws)
    torch.cuda.synchronize()
    return dict(dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(), dqb=dqb.cpu(), dkb=dkb.cpu(), dvb=dvb.cpu(),
                status=status, plan=plan, o=o_host, d_o=d_o_host)


def oracle_bwd(batch: wl.ThdBatch, res):
    z = lambda t: np.zeros(tuple(t.shape))
    return ob.thd_attention_bwd(as_f64(batch.q), as_f64(batch.k), as_f64(batch.v), as_f64(res["d_o"]),
                                batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.off_q, batch.off_k,
                                batch.off_v, batch.off_o, batch.mask_type, batch.q_causal_offset,
                                z(batch.q), z(batch.k), z(batch.v), softmax_scale=batch.softmax_scale,
                                window_left=batch.window_left)


def check_bwd(batch: wl.ThdBatch, res):
    dq_r, dk_r, dv_r, wq, wk, wv = oracle_bwd(batch, res)
    tol = TOL[batch.dtype]
    errs = {}
    for name, got, ref, w in (("dq", res["dq"], dq_r, wq), ("dk", res["dk"], dk_r, wk), ("dv", res["dv"], dv_r, wv)):
        g = got.to(torch.float64).numpy()[w]
        r = ref[w]
        assert np.isfinite(g).all(), f"non-finite {name} in a written row"
        err = float(np.max(np.abs(g - r), initial=0.0)) / max(1.0, float(np.max(np.abs(r), initial=0.0)))
        errs[name] = err
        assert err <= tol, f"{name} normalised error {err} > {tol}"
    # rows outside the sequences and token gaps keep the sentinel
    for name, back, w, h in (("dq", res["dqb"], wq, batch.h_q), ("dk", res["dkb"], wk, batch.h_kv),
                             ("dv", res["dvb"], wv, batch.h_kv)):
        raw = back.view(torch.uint8).numpy().reshape(back.shape[0], -1)
        assert (raw[~w] == SENTINEL).all(), f"a pad row of {name} was written"
        assert (raw[w][:, h * batch.d * back.element_size():] == SENTINEL).all(), f"{name} token gap written"
    return errs


SMALL = {
    "tiny_padded": {},
    "padded_causal": dict(b=4, h=4, min_len=64, max_len=400),
    "mixed_gqa": dict(b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2),
    "separate_padding": dict(b=6, max_len=500, h=4),
    "cp_chunks": dict(docs=2, k_len=1024, q_len=384, h=2),
}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_bwd_workloads_small(name, kernel):
    batch = wl.make(name, **SMALL[name])
    res = run_bwd(batch, kernel=kernel, seed=11)
    assert res["status"] == 0
    if kernel == bd.KERNEL_AUTO and batch.dtype in ("bf16", "fp16") and batch.d in (64, 128):
        assert res["plan"].kernel == bd.KERNEL_TCGEN05
    check_bwd(batch, res)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("windows", [None, (300, 0, 1000)])
def test_bwd_long_sequences(kernel, windows):
    """Sequences of many 128-row tiles on both axes (causal, so the per-unit tile
    ranges differ row to row and key to key), with and without windows."""
    batch = wl.padded_causal(b=3, h=2, min_len=900, max_len=1700)
    if windows is not None:
        batch = dataclasses.replace(batch, window_left=np.array(windows, dtype=np.int32))
    res = run_bwd(batch, kernel=kernel, seed=12)
    assert res["status"] == 0
    check_bwd(batch, res)


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_gqa_groups_tc(d):
    """Query-head groups of 4 summed into each kv head's dK/dV by the key-tile kernel."""
    batch = wl.random_pack(7100 + d, batch=4, max_len=600, h_q=8, h_kv=2, d=d, dtype="bf16",
                           allow_empty=False)
    res = run_bwd(batch, kernel=bd.KERNEL_TCGEN05, seed=13)
    assert res["status"] == 0
    check_bwd(batch, res)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("seed", range(8))
def test_bwd_random_packs(seed, kernel):
    """Ragged packs with mixed masks, causal offsets, windows, GQA, both Stats
    layouts and per-tensor token gaps on all eight views."""
    rng = np.random.default_rng(5000 + seed)
    dtype = ["bf16", "fp16", "fp32"][seed % 3]
    d = [64, 128, 32, 16][seed % 4]
    h_kv = int(rng.integers(1, 3))
    h_q = h_kv * int(rng.integers(1, 4))
    batch = wl.random_pack(6000 + seed, batch=int(rng.integers(1, 6)), max_len=int(rng.integers(1, 500)),
                           h_q=h_q, h_kv=h_kv, d=d, dtype=dtype, with_window=bool(seed % 2))
    gaps = tuple(int(x) for x in rng.integers(0, 3, size=8))
    res = run_bwd(batch, kernel=kernel, gaps=gaps, seed=seed)
    assert res["status"] == 0
    check_bwd(batch, res)


def test_bwd_empty_sequences_and_dead_rows():
    """Sequences with no queries still write dK = dV = 0 for their keys; rows with
    no visible key write dQ = 0."""
    # seed chosen so that sequence 4 has 0 queries and 54 keys, and negative causal
    # offsets leave the first rows of sequences 0, 1 and 3 without a visible key
    batch = wl.random_pack(7032, batch=5, max_len=90, h_q=2, h_kv=1, d=64, dtype="bf16", masks=(2,),
                           with_qco=True)
    assert batch.lens_q()[4] == 0 and batch.lens_k()[4] > 0 and batch.q_causal_offset[0] < 0
    res = run_bwd(batch, seed=3)
    assert res["status"] == 0
    check_bwd(batch, res)
    k0, n = int(batch.off_k[4]), int(batch.lens_k()[4])
    assert (res["dk"][k0:k0 + n].float() == 0).all() and (res["dv"][k0:k0 + n].float() == 0).all()
    q0 = int(batch.off_q[0])
    dead = -int(batch.q_causal_offset[0])           # rows i < -c see no key
    assert (res["dq"][q0:q0 + dead].float() == 0).all()


def test_bwd_invalid_sequence_flagged_and_untouched():
    batch = wl.random_pack(7002, batch=4, max_len=100, h_q=2, h_kv=2, d=64, dtype="bf16", allow_empty=False)
    mask = batch.mask_type.copy()
    mask[1] = 5
    res = run_bwd(batch, seed=4, device_mask=mask)
    assert res["status"] & bd.DEV_BAD_MASK
    # the bad sequence's gradient rows keep the sentinel
    for key, off, n in (("dqb", batch.off_q[1], batch.lens_q()[1]), ("dkb", batch.off_k[1], batch.lens_k()[1]),
                        ("dvb", batch.off_v[1], batch.lens_k()[1])):
        raw = res[key].view(torch.uint8).numpy().reshape(res[key].shape[0], -1)
        assert (raw[off:off + n] == SENTINEL).all()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("mult", [0, 2])
def test_bwd_element_offsets(kernel, mult):
    """Element-unit offsets (row x the primal tensor's token stride, over the
    multiplier) give the same gradients as row offsets; gradient views keep their
    own strides (token gaps)."""
    batch = wl.random_pack(7400 + mult, batch=4, max_len=300, h_q=4, h_kv=2, d=64, dtype="bf16",
                           stats_layout=wl.STATS_TOKEN_MAJOR)
    res = run_bwd(batch, kernel=kernel, gaps=(1, 0, 1, 0, 2, 1, 0, 2), seed=17, element_mult=mult)
    assert res["status"] == 0
    check_bwd(batch, res)


def _bwd_after_fwd(batch: wl.ThdBatch, kernel=bd.KERNEL_AUTO, seed=21, device="cuda"):
    # the forward always takes the automatic choice, so that two backward kernels
    # compared with each other read the same O and Stats
    """The benchmark's launch configuration: packed views, O and Stats from this
    library's forward on the same inputs (they are inputs of the backward, not of
    the oracle, which recomputes P from Q and K), dO seeded with NaN pad rows,
    gradient buffers filled with the byte sentinel."""
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(device)
    q, k, v = (t.to(device) for t in (batch.q, batch.k, batch.v))
    o = batch.o_init().to(device)
    stats = torch.zeros((batch.stats_numel,), dtype=torch.float32, device=device)
    d_o = _dout(batch, seed).to(device)
    cu_q, cu_k = ints(batch.cu_seqlens_q), ints(batch.cu_seqlens_kv)
    offs = [ints(x) for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o, batch.off_s)]
    mask = ints(batch.mask_type, np.int8)
    qco = None if batch.q_causal_offset is None else ints(batch.q_causal_offset)
    fplan = bd.plan_for_tensors(q, k, v, o, batch.batch, batch.cap_s, batch.stats_layout, batch.softmax_scale)
    fws = bd.alloc_workspace(fplan, device)
    bd.thd_attn_fwd(fplan, q, k, v, o, stats, cu_q, cu_k, *offs, mask, qco, fws)
    assert bd.thd_attn_read_status(fplan, fws) == 0
    grads = [torch.empty_like(t) for t in (q, k, v)]
    for g in grads:
        g.view(torch.uint8).fill_(SENTINEL)
    dq, dk, dv = grads
    plan = bd.plan_bwd_for_tensors(q, k, v, o, d_o, dq, dk, dv, batch.batch, batch.cap_s, batch.stats_layout,
                                   batch.softmax_scale, kernel, 0)
    ws = bd.alloc_workspace(plan, device)
    bd.thd_attn_bwd(plan, q, k, v, o, d_o, stats, dq, dk, dv, cu_q, cu_k, *offs, mask, qco, None, ws)
    status = bd.thd_attn_read_status(plan, ws)
    torch.cuda.synchronize()
    return dict(dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(), d_o=d_o.cpu(), status=status, plan=plan)


def _check_group(batch: wl.ThdBatch, res, b: int, g: int):
    """Every row of sequence ``b``'s dQ (query heads of kv group ``g``) and of its
    dK / dV at kv head ``g`` against the oracle, one query head at a time."""
    from oracle.thd_attention import causal_shift
    lq, lk = int(batch.lens_q()[b]), int(batch.lens_k()[b])
    qs, ks, vs, os_ = (int(x[b]) for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o))
    shift = causal_shift(int(batch.mask_type[b]), lq, lk,
                         None if batch.q_causal_offset is None else batch.q_causal_offset[b])
    scale = batch.softmax_scale if batch.softmax_scale is not None else 1.0 / np.sqrt(batch.d)
    group = batch.h_q // batch.h_kv
    f64 = lambda t: t.to(torch.float64).numpy()
    kb, vb = f64(batch.k[ks:ks + lk, g]), f64(batch.v[vs:vs + lk, g])
    acc_k, acc_v = np.zeros_like(kb), np.zeros_like(vb)
    tol = TOL[batch.dtype]

    def close(name, got, ref):
        assert np.isfinite(got).all(), f"non-finite {name}"
        err = float(np.max(np.abs(got - ref), initial=0.0)) / max(1.0, float(np.max(np.abs(ref), initial=0.0)))
        assert err <= tol, f"seq {b} group {g} {name}: normalised error {err} > {tol}"

    for h in range(g * group, (g + 1) * group):
        gq, gk, gv = ob.attention_one_head_bwd(f64(batch.q[qs:qs + lq, h]), kb, vb,
                                               f64(res["d_o"][os_:os_ + lq, h]), scale, shift)
        close(f"dq head {h}", f64(res["dq"][qs:qs + lq, h]), gq)
        acc_k += gk
        acc_v += gv
    close("dk", f64(res["dk"][ks:ks + lk, g]), acc_k)
    close("dv", f64(res["dv"][vs:vs + lk, g]), acc_v)


def _written_rows(offs, lens, cap):
    w = np.zeros(cap, dtype=bool)
    for o, n in zip(offs, lens):
        w[int(o):int(o) + int(n)] = True
    return w


def _check_dq_rows(batch: wl.ThdBatch, res, b: int, rows, heads):
    """dQ of single query rows: row i's gradient depends on row i alone, so a
    one-row problem with the row's own causal shift gives it exactly."""
    from oracle.thd_attention import causal_shift
    lq, lk = int(batch.lens_q()[b]), int(batch.lens_k()[b])
    qs, ks, vs, os_ = (int(x[b]) for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o))
    shift = causal_shift(int(batch.mask_type[b]), lq, lk,
                         None if batch.q_causal_offset is None else batch.q_causal_offset[b])
    scale = batch.softmax_scale if batch.softmax_scale is not None else 1.0 / np.sqrt(batch.d)
    group = batch.h_q // batch.h_kv
    f64 = lambda t: t.to(torch.float64).numpy()
    tol = TOL[batch.dtype]
    for h in heads:
        g = h // group
        kb, vb = f64(batch.k[ks:ks + lk, g]), f64(batch.v[vs:vs + lk, g])
        for r in rows:
            gq, _, _ = ob.attention_one_head_bwd(f64(batch.q[qs + r:qs + r + 1, h]), kb, vb,
                                                 f64(res["d_o"][os_ + r:os_ + r + 1, h]), scale,
                                                 None if shift is None else shift + r)
            got = f64(res["dq"][qs + r:qs + r + 1, h])
            err = float(np.max(np.abs(got - gq))) / max(1.0, float(np.max(np.abs(gq))))
            assert err <= tol, f"seq {b} row {r} head {h}: dq normalised error {err} > {tol}"


def _check_dv_sums(batch: wl.ThdBatch, res, b: int):
    """An identity of the softmax gradient that holds at any size, per kv head g:
    sum_j dV_j = sum of dO_i over the group's heads and the live rows (every live
    row of P sums to one), so it checks the Stats each key tile reads. Tolerance
    2e-2 of max(1, |sum dO|): 16-bit rounding of the stored dV moves the sum by at
    most 2^-8 of sum_i |dO_i| and by far less in practice, a misread Stats row by
    a factor. (The companion identity sum_j dK_j = 0 has no usable bound here: the
    16-bit dS rounding is not small against the cancelling sum.)"""
    from oracle.thd_attention import causal_shift
    lq, lk = int(batch.lens_q()[b]), int(batch.lens_k()[b])
    vs, os_ = int(batch.off_v[b]), int(batch.off_o[b])
    shift = causal_shift(int(batch.mask_type[b]), lq, lk,
                         None if batch.q_causal_offset is None else batch.q_causal_offset[b])
    n_vis = np.full(lq, lk) if shift is None else np.clip(np.arange(lq) + shift + 1, 0, lk)
    live = torch.from_numpy(n_vis > 0)
    group = batch.h_q // batch.h_kv
    d_o = res["d_o"][os_:os_ + lq][live].to(torch.float64)                      # [live, h_q, d]
    want = d_o.view(-1, batch.h_kv, group, batch.d).sum(dim=(0, 2))            # [h_kv, d]
    got = res["dv"][vs:vs + lk].to(torch.float64).sum(dim=0)
    err = float((got - want).abs().max()) / max(1.0, float(want.abs().max()))
    assert err <= 2e-2, f"seq {b}: sum of dV rows off by {err}"


@pytest.mark.parametrize("name", ["cp_chunks", "mixed_gqa"])
def test_bwd_full_size_sampled(name):
    """Full-size workloads in the benchmark's launch configuration. cp_chunks: dQ of
    sampled rows of both documents at three heads against the oracle (one whole
    65536-key head costs the oracle about a minute, so dK and dV are checked through
    the dV row-sum identity and against the SIMT kernel); mixed_gqa: every row of
    the longest sequence and two others at sampled kv groups. Both: the identity on
    every sequence, pad rows untouched, every row against the SIMT backward."""
    batch = wl.make(name)
    res = _bwd_after_fwd(batch)
    assert res["status"] == 0
    assert res["plan"].kernel == bd.KERNEL_TCGEN05
    lq, lk = batch.lens_q(), batch.lens_k()
    rng = np.random.default_rng(3)
    if name == "cp_chunks":
        for b in range(batch.batch):
            L = int(lq[b])
            rows = sorted({0, 1, 127, 128, 129, 255, 256, L - 2, L - 1, *rng.integers(0, L, size=3).tolist()})
            _check_dq_rows(batch, res, b, rows, heads=(0, batch.h_q // 2 - 1, batch.h_q - 1))
    else:
        longest = int(np.argmax(lq))
        others = [int(x) for x in rng.choice(np.nonzero(lq > 0)[0], size=3, replace=False) if x != longest][:2]
        pairs = [(longest, 0), (longest, batch.h_kv - 1)] + [(b, int(rng.integers(batch.h_kv))) for b in others]
        for b, g in pairs:
            _check_group(batch, res, b, g)
    for b in range(batch.batch):
        _check_dv_sums(batch, res, b)
    for key, offs, lens in (("dq", batch.off_q, lq), ("dk", batch.off_k, lk), ("dv", batch.off_v, lk)):
        raw = res[key].view(torch.uint8).numpy().reshape(res[key].shape[0], -1)
        w = _written_rows(offs, lens, raw.shape[0])
        assert (raw[~w] == SENTINEL).all(), f"a pad row of {key} was written"
    alt = _bwd_after_fwd(batch, kernel=bd.KERNEL_SIMT)
    assert alt["status"] == 0
    for key, offs, lens in (("dq", batch.off_q, lq), ("dk", batch.off_k, lk), ("dv", batch.off_v, lk)):
        w = torch.from_numpy(_written_rows(offs, lens, res[key].shape[0]))
        a, r = res[key][w].float(), alt[key][w].float()
        err = float((a - r).abs().max()) / max(1.0, float(r.abs().max()))
        assert err <= 2 * TOL[batch.dtype], f"{key}: tcgen05 vs SIMT normalised error {err}"


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("d,h_q,h_kv", [(128, 4, 2), (64, 2, 2)])
def test_bwd_zigzag_chunks_share_keys(kernel, d, h_q, h_kv):
    """The zigzag query chunks of two documents (Megatron-LM PR #14: under context
    parallelism rank r holds chunks r and 2*cp-1-r of each document): four segments
    per document read the SAME K/V rows, each bottom-right over the key prefix that
    ends with its chunk. dK / dV of a shared row is the sum over the segments that
    see it, written once; against the oracle, which sums them."""
    batch = wl.zigzag_chunks(docs=2, doc_len=2048, h_q=h_q, h_kv=h_kv, d=d)
    res = run_bwd(batch, kernel=kernel, seed=31)
    assert res["status"] == 0
    if kernel == bd.KERNEL_AUTO:
        assert res["plan"].kernel == bd.KERNEL_TCGEN05
    check_bwd(batch, res)


def _shifted_k(batch: wl.ThdBatch, order=None, shift=None):
    """The batch with its K/V rows laid out per ``order`` (a permutation of the
    sequences, packed with one gap row) and sequence ``shift[0]`` moved by
    ``shift[1]`` rows (into its neighbour's rows when that is negative)."""
    lk = batch.lens_k()
    order = list(range(batch.batch)) if order is None else order
    off = np.zeros(batch.batch + 1, dtype=np.int64)
    pos = 0
    for b in order:
        off[b] = pos
        pos += int(lk[b]) + 1
    off[batch.batch] = pos
    if shift is not None:
        off[shift[0]] += shift[1]
    k = torch.zeros((pos, batch.h_kv, batch.d), dtype=batch.torch_dtype)
    v = torch.zeros_like(k)
    for b in range(batch.batch):
        n = int(lk[b])
        k[off[b]:off[b] + n] = batch.k[batch.off_k[b]:batch.off_k[b] + n]
        v[off[b]:off[b] + n] = batch.v[batch.off_v[b]:batch.off_v[b] + n]
    off = off.astype(np.int32)
    return dataclasses.replace(batch, k=k, v=v, off_k=off, off_v=off.copy())


@pytest.mark.parametrize("kernel", KERNELS)
def test_bwd_unsorted_key_rows(kernel):
    """Key rows laid out in reverse sequence order (disjoint): the overlap check
    compares every pair of sequences and finds nothing; gradients exact."""
    batch = wl.random_pack(7300, batch=5, max_len=200, h_q=2, h_kv=1, d=64, dtype="bf16", allow_empty=False)
    batch = _shifted_k(batch, order=list(range(batch.batch))[::-1])
    res = run_bwd(batch, kernel=kernel, seed=32)
    assert res["status"] == 0
    check_bwd(batch, res)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("unsorted", [False, True])
def test_bwd_partial_key_overlap_flagged(kernel, unsorted):
    """Two sequences whose K/V rows partly overlap without being one key group: the
    status word reports THD_DEV_KEY_OVERLAP, no dK / dV row is written, dQ is
    still exact."""
    batch = wl.random_pack(7301, batch=4, max_len=200, h_q=2, h_kv=1, d=64, dtype="bf16", allow_empty=False)
    order = [3, 2, 1, 0] if unsorted else None
    # sequence 2 starts 5 rows before its own rows: inside sequence 1's (or, in
    # reverse order, sequence 3's) last rows
    batch = _shifted_k(batch, order=order, shift=(2, -5))
    res = run_bwd(batch, kernel=kernel, seed=33)
    assert res["status"] & bd.DEV_KEY_OVERLAP
    dq_r, _, _, wq, _, _ = oracle_bwd(batch, res)
    g = res["dq"].to(torch.float64).numpy()[wq]
    err = float(np.max(np.abs(g - dq_r[wq]))) / max(1.0, float(np.max(np.abs(dq_r[wq]))))
    assert err <= TOL[batch.dtype]
    for key in ("dkb", "dvb"):
        assert (res[key].view(torch.uint8).numpy() == SENTINEL).all(), f"{key} written despite the overlap"


def test_bwd_full_size_every_row_mixed_gqa():
    """The full-size mixed-policy GQA workload in the benchmark's launch configuration
    (O and Stats from this library's forward): dQ, dK and dV of every row and head
    against the backward oracle (normalised max error per gradient, as elsewhere),
    and every row outside the sequences untouched."""
    batch = wl.make("mixed_gqa")
    res = _bwd_after_fwd(batch)
    assert res["status"] == 0
    assert res["plan"].kernel == bd.KERNEL_TCGEN05
    dq_r, dk_r, dv_r, wq, wk, wv = oracle_bwd(batch, res)
    tol = TOL[batch.dtype]
    for name, got, ref, w in (("dq", res["dq"], dq_r, wq), ("dk", res["dk"], dk_r, wk), ("dv", res["dv"], dv_r, wv)):
        g = got.to(torch.float64).numpy()[w]
        r = ref[w]
        assert np.isfinite(g).all(), f"non-finite {name}"
        err = float(np.max(np.abs(g - r))) / max(1.0, float(np.max(np.abs(r))))
        assert err <= tol, f"{name}: normalised error {err} > {tol}"
        raw = got.view(torch.uint8).numpy().reshape(got.shape[0], -1)
        assert (raw[~w] == SENTINEL).all(), f"a row of {name} outside the sequences was written"
