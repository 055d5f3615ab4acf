"""Guard bands around every buffer an entry point writes.

The bug class behind NVIDIA/cudnn-frontend PR #462 is a ragged backward whose
workspace was sized too small and overwritten past its end ("Why this was never
caught": the suite's guard-band check, "workspace overwritten outside its
boundaries"). Here each workspace (exactly ``workspace_bytes`` long, not rounded
up) and each output buffer sits between two 64 KiB regions filled with a byte
pattern; after the call, with the device synchronised, every byte of both regions
must still hold it. The entry points run at full size in the benchmark's launch
configuration: the forward with and without the key-range split (whose fp32
partial results live in the workspace), the backward (its (LSE, D) blocks and
second schedule), the indexer top-k (a float32 score row per output row), on the
128k-token context-parallel chunks, on the separate-padding workload with
head-major Stats, and at the head-major Stats shape with strides
(58880, 7360, 1, 1) that the PR page prints.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GUARD = 64 * 1024
PATTERN = 0x3C


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


class Guarded:
    """Buffers carved out of larger allocations with a guard region on each side."""

    def __init__(self, device="cuda"):
        self.device = device
        self.blocks: list[tuple[str, torch.Tensor, int]] = []

    def bytes(self, name: str, nbytes: int) -> torch.Tensor:
        """``nbytes`` of device memory, 256-byte aligned, guards right at both ends."""
        big = torch.empty(GUARD + nbytes + GUARD, dtype=torch.uint8, device=self.device)
        big.fill_(PATTERN)
        self.blocks.append((name, big, nbytes))
        return big[GUARD:GUARD + nbytes]

    def like(self, name: str, src: torch.Tensor, fill_byte: int | None = None) -> torch.Tensor:
        """A contiguous device copy of ``src`` (or a buffer of its shape filled with
        ``fill_byte``) inside guards."""
        n = src.numel() * src.element_size()
        raw = self.bytes(name, n)
        t = raw.view(src.dtype).view(src.shape)
        if fill_byte is None:
            t.copy_(src)
        else:
            raw.fill_(fill_byte)
        return t

    def workspace(self, plan) -> torch.Tensor:
        return self.bytes("workspace", max(1, plan.workspace_bytes))

    def check(self):
        torch.cuda.synchronize()
        for name, big, n in self.blocks:
            head = big[:GUARD]
            tail = big[GUARD + n:]
            assert bool((head == PATTERN).all()), f"{name}: the guard before the buffer was written"
            assert bool((tail == PATTERN).all()), f"{name}: the guard after the buffer was written"


def _ints(a, dev, dt=np.int32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)


def _fwd(batch: wl.ThdBatch, g: Guarded, flags=0):
    dev = g.device
    q, k, v = g.like("q", batch.q), g.like("k", batch.k), g.like("v", batch.v)
    o = g.like("o", batch.o_init())
    stats = g.like("stats", batch.stats_init())
    meta = [_ints(x, dev) for x in (batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.off_q, batch.off_k,
                                    batch.off_v, batch.off_o, batch.off_s)]
    mask = _ints(batch.mask_type, dev, np.int8)
    qco = None if batch.q_causal_offset is None else _ints(batch.q_causal_offset, dev)
    plan = bd.plan_for_tensors(q, k, v, o, batch.batch, batch.cap_s, batch.stats_layout,
                               batch.softmax_scale, bd.KERNEL_AUTO, flags)
    ws = g.workspace(plan)
    bd.thd_attn_fwd(plan, q, k, v, o, stats, *meta, mask, qco, ws)
    assert bd.thd_attn_read_status(plan, ws) == 0
    return dict(q=q, k=k, v=v, o=o, stats=stats, meta=meta, mask=mask, qco=qco, plan=plan)


def _bwd(batch: wl.ThdBatch, g: Guarded):
    f = _fwd(batch, g)
    gen = torch.Generator().manual_seed(5)
    d_o = g.like("d_o", torch.randn((batch.cap_o, batch.h_q, batch.d), generator=gen).to(batch.torch_dtype))
    dq = g.like("dq", batch.q, fill_byte=wl.SENTINEL_BYTE)
    dk = g.like("dk", batch.k, fill_byte=wl.SENTINEL_BYTE)
    dv = g.like("dv", batch.v, fill_byte=wl.SENTINEL_BYTE)
    plan = bd.plan_bwd_for_tensors(f["q"], f["k"], f["v"], f["o"], d_o, dq, dk, dv, batch.batch, batch.cap_s,
                                   batch.stats_layout, batch.softmax_scale)
    assert plan.kernel == bd.KERNEL_TCGEN05
    ws = g.workspace(plan)
    bd.thd_attn_bwd(plan, f["q"], f["k"], f["v"], f["o"], d_o, f["stats"], dq, dk, dv, *f["meta"], f["mask"],
                    f["qco"], None, ws)
    assert bd.thd_attn_read_status(plan, ws) == 0


def _head_major(batch: wl.ThdBatch) -> wl.ThdBatch:
    return dataclasses.replace(batch, stats_layout=wl.STATS_HEAD_MAJOR)


def _stats_7360() -> wl.ThdBatch:
    """Head-major Stats of 8 heads over 7360 rows: strides (58880, 7360, 1, 1) as
    [B=1, H, T, 1]; the packed sequences end near the Stats capacity."""
    batch = wl.padded_causal(seed=462, b=12, h=8, min_len=300, max_len=900)
    assert int(batch.off_s[-1]) <= 7360
    batch = dataclasses.replace(batch, stats_layout=wl.STATS_HEAD_MAJOR, cap_s=7360)
    assert batch.stats_strides == (1, 7360) and batch.h_q * batch.cap_s == 58880
    return batch


@pytest.mark.parametrize("flags", [0, bd.FLAG_NO_KV_SPLIT])
def test_guards_fwd_cp_chunks(flags):
    g = Guarded()
    f = _fwd(wl.cp_chunks(), g, flags)
    if flags == 0:
        assert f["plan"].workspace_bytes > 64 * 1024 * 1024, "the split's partial buffers are in the workspace"
    g.check()


@pytest.mark.parametrize("make", [lambda: _head_major(wl.separate_padding()), _stats_7360],
                         ids=["separate_padding_head_major", "stats_58880_7360"])
def test_guards_fwd_head_major(make):
    g = Guarded()
    _fwd(make(), g)
    g.check()


@pytest.mark.parametrize("make", [wl.cp_chunks, lambda: _head_major(wl.separate_padding()), _stats_7360],
                         ids=["cp_chunks", "separate_padding_head_major", "stats_58880_7360"])
def test_guards_bwd(make):
    g = Guarded()
    _bwd(make(), g)
    g.check()


@pytest.mark.parametrize("make", [wl.indexer_cp, wl.indexer_zigzag], ids=["indexer_cp", "indexer_zigzag"])
def test_guards_indexer(make):
    batch = make()
    g = Guarded()
    dev = g.device
    q, k, w = g.like("qi", batch.q), g.like("ki", batch.k), g.like("w", batch.w)
    idx = g.like("idx", torch.empty((batch.cap_out, batch.topk), dtype=torch.int32), fill_byte=0x7F)
    sc = g.like("scores", torch.empty((batch.cap_out, batch.topk), dtype=torch.float32), fill_byte=0x7F)
    mask = _ints(batch.mask_type, dev, np.int8)
    qco = None if batch.q_causal_offset is None else _ints(batch.q_causal_offset, dev)
    max_k = int(batch.lens_k().max())
    plan = bd.indexer_plan_for_tensors(q, k, w, idx, batch.batch, batch.topk, max_k)
    ws = g.workspace(plan)
    bd.thd_indexer_topk(plan, q, k, w, idx, sc, _ints(batch.cu_seqlens_q, dev), _ints(batch.cu_seqlens_kv, dev),
                        _ints(batch.off_q, dev), _ints(batch.off_k, dev), _ints(batch.off_out, dev), mask, qco, ws)
    assert bd.thd_attn_read_status(plan, ws) == 0
    g.check()
