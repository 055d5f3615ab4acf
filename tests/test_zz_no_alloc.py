"""The workspace-free entry point, for callers that cannot allocate device memory
where they run attention (during CUDA-graph capture, inside runtimes that own all
device memory, in latency-critical loops). Its calls must give the same bytes as
the regular entry point with a caller workspace, call after call and after a call
on a different plan has left other contents in the shared static array, while the
library allocates no device memory. Collected last on purpose: if it fails, a run
that stops at the first failure has already run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


def _device_batch(batch, dev):
    ints = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)
    return dict(q=batch.q.to(dev), k=batch.k.to(dev), v=batch.v.to(dev),
                meta=[ints(batch.cu_seqlens_q), ints(batch.cu_seqlens_kv), ints(batch.off_q),
                      ints(batch.off_k), ints(batch.off_v), ints(batch.off_o), ints(batch.off_s),
                      ints(batch.mask_type, np.int8)],
                qco=None if batch.q_causal_offset is None else ints(batch.q_causal_offset))


def _plan(batch, d, o):
    # the static array holds no partial results of split key ranges: plan without splitting
    plan = bd.plan_for_tensors(d["q"], d["k"], d["v"], o, batch.batch, batch.cap_s, batch.stats_layout,
                               flags=bd.FLAG_NO_KV_SPLIT)
    assert plan.workspace_bytes <= bd.static_workspace_capacity()
    return plan


def _outputs(batch, dev):
    return batch.o_init().to(dev), batch.stats_init().to(dev)


def _static_call(batch, d, plan, out=None):
    o, s = _outputs(batch, d["q"].device) if out is None else out
    bd.thd_attn_fwd_static_ws(plan, d["q"], d["k"], d["v"], o, s, *d["meta"], d["qco"])
    return o, s


CASES = [
    ("mixed_gqa", dict(b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2)),
    ("separate_padding", dict(b=6, max_len=500, h=4)),
    ("tiny_padded", {}),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_static_workspace_matches_workspace_entry(name, kw):
    dev = torch.device("cuda", 0)
    batch = wl.make(name, **kw)
    d = _device_batch(batch, dev)
    o_ref = batch.o_init().to(dev)
    s_ref = batch.stats_init().to(dev)
    plan = _plan(batch, d, o_ref)
    ws = bd.alloc_workspace(plan, dev)
    bd.thd_attn_fwd(plan, d["q"], d["k"], d["v"], o_ref, s_ref, *d["meta"], d["qco"], ws)
    assert bd.thd_attn_read_status(plan, ws) == 0
    # a different plan and batch (more sequences, other lengths and offsets) whose call
    # leaves its own header, metadata and tile list in the shared array in between
    other = wl.make("mixed_gqa", b=9, median=96, max_len=900, total=2600, h_q=4, h_kv=4, seed=7)
    d2 = _device_batch(other, dev)
    plan2 = _plan(other, d2, other.o_init().to(dev))
    # every output buffer exists before the memory counters are read
    outs = [_outputs(batch, dev) for _ in range(2)]
    other_out = _outputs(other, dev)
    # the first static call on this device resolves the array's address (and may load
    # the module); the device memory in use must not change after it
    _static_call(batch, d, plan, _outputs(batch, dev))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for call in range(2):
        _static_call(batch, d, plan, outs[call])
        assert bd.thd_attn_static_read_status(plan) == 0
        if call == 0:
            _static_call(other, d2, plan2, other_out)
            assert bd.thd_attn_static_read_status(plan2) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0, "device memory changed across the static calls"
    assert torch.cuda.memory_allocated(dev) == alloc0
    for call, (o, s) in enumerate(outs):
        # same kernels on the same schedule as the workspace entry: identical bytes,
        # pad rows included (they keep the sentinel in both)
        assert torch.equal(o.view(torch.uint8), o_ref.view(torch.uint8)), f"call {call}: O bytes differ"
        assert torch.equal(s.view(torch.int32), s_ref.view(torch.int32)), f"call {call}: Stats bytes differ"


def test_static_workspace_allocates_nothing():
    """With the output buffers made beforehand, repeated static calls change neither
    torch's allocator counters nor the device's free memory."""
    dev = torch.device("cuda", 0)
    batch = wl.make("mixed_gqa", b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2)
    d = _device_batch(batch, dev)
    o = batch.o_init().to(dev)
    s = batch.stats_init().to(dev)
    plan = _plan(batch, d, o)
    bd.thd_attn_fwd_static_ws(plan, d["q"], d["k"], d["v"], o, s, *d["meta"], d["qco"])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    stats0 = torch.cuda.memory_stats(dev)
    for _ in range(3):
        bd.thd_attn_fwd_static_ws(plan, d["q"], d["k"], d["v"], o, s, *d["meta"], d["qco"])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    stats1 = torch.cuda.memory_stats(dev)
    assert free1 == free0
    for key in ("allocation.all.allocated", "reserved_bytes.all.allocated", "allocated_bytes.all.allocated"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


def test_static_status_reports_bad_offset():
    """A sequence whose K rows lie past the view's capacity is reported through the
    static array's status word and gets no work; the other sequences are exact."""
    dev = torch.device("cuda", 0)
    batch = wl.random_pack(5, batch=5, max_len=100, h_q=2, h_kv=2, d=64, dtype="bf16", allow_empty=False)
    bad = wl.ThdBatch(**{**batch.__dict__})
    bad.off_k = batch.off_k.copy()
    bad.off_k[1] = batch.k.shape[0]
    d = _device_batch(bad, dev)
    o_ref = bad.o_init().to(dev)
    s_ref = bad.stats_init().to(dev)
    plan = _plan(bad, d, o_ref)
    ws = bd.alloc_workspace(plan, dev)
    bd.thd_attn_fwd(plan, d["q"], d["k"], d["v"], o_ref, s_ref, *d["meta"], d["qco"], ws)
    assert bd.thd_attn_read_status(plan, ws) == bd.DEV_BAD_OFFSET
    o, s = _static_call(bad, d, plan)
    assert bd.thd_attn_static_read_status(plan) == bd.DEV_BAD_OFFSET
    assert torch.equal(o.view(torch.uint8), o_ref.view(torch.uint8))
    assert torch.equal(s.view(torch.int32), s_ref.view(torch.int32))
    # a valid call afterwards clears the word again
    good = _device_batch(batch, dev)
    _static_call(batch, good, plan)
    assert bd.thd_attn_static_read_status(plan) == 0


def test_static_workspace_rejects_oversized_plan():
    cap = bd.static_workspace_capacity()
    # a plan whose metadata alone exceeds the static array: 32 bytes per sequence
    batch = cap // 32 + 1
    desc = bd.make_desc(torch.bfloat16, batch, 1, 1, 64, (1, 1, 1, 1), (64, 64, 64, 64), (64, 64, 64, 64),
                        cap_rows_stats=1)
    plan = bd.thd_attn_plan(desc)
    assert plan.workspace_bytes > cap
    with pytest.raises(bd.ThdAttnError) as e:
        bd.thd_attn_fwd_static_ws(plan, *([None] * 14))
    assert e.value.status == 5
