"""The workspace-free entry point, for callers that cannot allocate device memory
where they run attention (during CUDA-graph capture, inside runtimes that own all
device memory, in latency-critical loops). It must give the same results as the
regular entry point with a caller workspace, call after call, while the library
allocates nothing. Collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl
from tests.gpu_harness import TOL

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


@pytest.mark.parametrize("name,kw", [
    ("mixed_gqa", dict(b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2)),
    ("separate_padding", dict(b=6, max_len=500, h=4)),
    ("tiny_padded", {}),
])
def test_static_workspace_matches_workspace_entry(name, kw):
    dev = torch.device("cuda", 0)
    batch = wl.make(name, **kw)
    d = _device_batch(batch, dev)
    o_ref = batch.o_init().to(dev)
    s_ref = batch.stats_init().to(dev)
    # the static array holds no partial results of split key ranges: plan without splitting
    plan = bd.plan_for_tensors(d["q"], d["k"], d["v"], o_ref, batch.batch, batch.cap_s, batch.stats_layout,
                               flags=bd.FLAG_NO_KV_SPLIT)
    assert plan.workspace_bytes <= bd.static_workspace_capacity()
    ws = bd.alloc_workspace(plan, dev)
    bd.thd_attn_fwd(plan, d["q"], d["k"], d["v"], o_ref, s_ref, *d["meta"], d["qco"], ws)
    assert bd.thd_attn_read_status(plan, ws) == 0
    tol_o, tol_l = TOL[batch.dtype]
    for call in range(2):
        o = batch.o_init().to(dev)
        s = batch.stats_init().to(dev)
        bd.thd_attn_fwd_static_ws(plan, d["q"], d["k"], d["v"], o, s, *d["meta"], d["qco"])
        torch.cuda.synchronize()
        a, b = o.float().cpu(), o_ref.float().cpu()
        same_nan = torch.equal(torch.isnan(a), torch.isnan(b))
        assert same_nan, f"call {call}: written rows differ"
        diff = torch.nan_to_num((a - b).abs(), nan=0.0)
        assert float(diff.max()) <= tol_o, f"call {call}: O differs by {float(diff.max())}"
        sa, sb = s.cpu(), s_ref.cpu()
        assert torch.equal(torch.isneginf(sa), torch.isneginf(sb))
        fin = torch.isfinite(sa) & torch.isfinite(sb)
        assert float((sa[fin] - sb[fin]).abs().max()) <= tol_l, f"call {call}: LSE differs"
        # pad rows stay untouched: the sentinel bytes of both outputs agree exactly
        assert torch.equal(o.cpu().view(torch.uint8) == wl.SENTINEL_BYTE,
                           o_ref.cpu().view(torch.uint8) == wl.SENTINEL_BYTE)


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
