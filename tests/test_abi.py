"""C-ABI checks that need no GPU: the library loads, exports every declared
entry point, validates descriptors on the host, and applies the all-axes span
rule for capacities."""
from __future__ import annotations

import ctypes
import json
import math
import os
import re

import pytest
import torch

import ragged_varlen_attention_gb300 as rva
from ragged_varlen_attention_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "thd_attn.h")


@pytest.fixture(scope="module")
def lib():
    from ragged_varlen_attention_gb300 import build
    build.build()
    return bd.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(thd_(?:attn|indexer)_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def _desc(**kw):
    base = dict(dtype=torch.bfloat16, batch=2, h_q=4, h_kv=2, d=128, cap_rows=(100, 80, 80, 100),
                stride_tok=(512, 256, 256, 512), stride_head=(128, 128, 128, 128), nbytes=(0, 0, 0, 0),
                cap_rows_stats=100, stats_layout=bd.STATS_TOKEN_MAJOR, softmax_scale=None,
                kernel=bd.KERNEL_AUTO)
    base.update(kw)
    return bd.make_desc(**base)


def _plan_status(desc):
    lib = bd.load_library()
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_attn_plan(ctypes.byref(h), ctypes.byref(desc), ctypes.byref(ws))
    if st == 0:
        lib.thd_attn_plan_destroy(h)
    return st, ws.value


def test_plan_accepts_valid(lib):
    st, ws = _plan_status(_desc())
    assert st == 0 and ws > 0 and ws % 256 == 0


@pytest.mark.parametrize("kw,code", [
    (dict(h_q=3, h_kv=2), 1),
    (dict(d=0), 1),
    (dict(d=160), 2),
    (dict(batch=-1), 1),
    (dict(cap_rows=(-1, 80, 80, 100)), 1),
    (dict(stride_tok=(-4, 256, 256, 512)), 1),
    (dict(stats_layout=5), 1),
    (dict(softmax_scale=math.inf), 1),
    (dict(kernel=9), 1),
    (dict(nbytes=(100 * 512 * 2 - 2, 0, 0, 0)), 4),      # one element short of the span
])
def test_plan_rejects(lib, kw, code):
    st, _ = _plan_status(_desc(**kw))
    assert st == code


def test_plan_capacity_exact_fit(lib):
    span = (99 * 512 + 3 * 128 + 127 + 1) * 2
    assert _plan_status(_desc(nbytes=(span, 0, 0, 0)))[0] == 0
    assert _plan_status(_desc(nbytes=(span - 1, 0, 0, 0)))[0] == 4


def test_span_rule_matches_page_closed_forms(lib):
    """cudnn-frontend PR #462 'The fix': for token-major inputs the all-axes span equals
    maxT*h_q (softmax_sum) and maxT*h_q*d (dQ_accum); head-major [h, t] stats span
    h_q*T_s."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "stats_layout.json")))
    span = lib.thd_attn_view_span_bytes
    for max_t, h_q, d in [(7, 3, 5), (1024, 16, 128), (7360, 8, 64)]:
        assert span(max_t, h_q, 1, h_q, 1, 1) == max_t * h_q
        assert span(max_t, h_q, d, h_q * d, d, 1) == max_t * h_q * d
    h_q, t = g["h_q"], g["t_capacity"]
    seq_stride, head_stride, tok_stride, _ = g["head_major_stats_strides"]
    assert span(t, h_q, 1, tok_stride, head_stride, 4) == seq_stride * 4
    # the under-sizing the page describes: sizing head-major stats from the token
    # stride alone (stride 1) misses a factor h_q
    assert span(t, 1, 1, tok_stride, 0, 4) * h_q == span(t, h_q, 1, tok_stride, head_stride, 4)
    assert span(0, 4, 4, 16, 4, 2) == 0


def test_kernel_selection(lib):
    p = bd.thd_attn_plan(_desc(dtype=torch.float32))
    assert p.kernel == bd.KERNEL_SIMT
    p = bd.thd_attn_plan(_desc(kernel=bd.KERNEL_SIMT))
    assert p.kernel == bd.KERNEL_SIMT
    p = bd.thd_attn_plan(_desc(d=96))
    assert p.kernel == bd.KERNEL_SIMT
    with pytest.raises(bd.ThdAttnError):
        bd.thd_attn_plan(_desc(d=96, kernel=bd.KERNEL_TCGEN05))
    # token stride not a multiple of 16 bytes: no TMA path
    with pytest.raises(bd.ThdAttnError):
        bd.thd_attn_plan(_desc(stride_tok=(520 + 4, 256, 256, 512), kernel=bd.KERNEL_TCGEN05))


def test_workspace_layout_counter_first(lib):
    p = bd.thd_attn_plan(_desc(batch=37))
    hdr, meta, base, pairs = p.workspace_layout
    assert hdr == 0 and meta >= 64 and base >= meta + 37 * 32 and pairs >= base + 38 * 4
    assert p.workspace_bytes >= pairs + p.max_pairs * 8
    assert all(x % 256 == 0 for x in p.workspace_layout)
    # capacity bound: every sequence may add one partial tile
    assert p.max_pairs >= 37 + math.ceil(100 / p.rows_per_unit)


def test_fwd_rejects_bad_workspace_without_touching_device(lib):
    p = bd.thd_attn_plan(_desc())
    nullp = ctypes.c_void_p(0)
    args = [ctypes.c_void_p(p.handle)] + [ctypes.c_void_p(256)] * 14 + [nullp, nullp]
    assert lib.thd_attn_fwd(*args) == 5            # workspace NULL
    args[15] = ctypes.c_void_p(4096 + 8)
    assert lib.thd_attn_fwd(*args) == 5            # workspace not 256-byte aligned
    assert lib.thd_attn_fwd(None, *args[1:]) == 1  # no plan


def test_status_strings(lib):
    for code in range(7):
        assert lib.thd_attn_status_string(code).decode().startswith("THD_")


def test_package_import_does_not_load_library():
    # importing the package is side-effect free; the binding loads the library lazily
    assert hasattr(rva, "thd_attn_forward")


def test_unit_order_covers_every_pair_and_head_once():
    """The work-id -> (pair, head) order of the schedule is a permutation that keeps
    the longest-first cost groups and puts query heads of one kv head innermost."""
    from tests import schedule_mirror as sm
    pairs = [(0, 0, 600), (1, 0, 300), (1, 256, 290), (2, 0, 3), (3, 0, 0)]
    starts = sm.group_starts(pairs)
    assert starts[0] == 0 and starts[-1] == len(pairs)
    order = sm.unit_order(starts, h_q=8, h_kv=2)
    assert sorted(order) == sorted((p, h) for p in range(len(pairs)) for h in range(8))
    # group of pair 0 (cost 600) first; inside group 1 (costs 256..511): kv head 0's
    # units (query heads 0-3) for pairs 1 and 2 before kv head 1's
    assert order[:8] == [(0, h) for h in range(4)] + [(0, h) for h in range(4, 8)]
    assert order[8:16] == [(1, 0), (1, 1), (1, 2), (1, 3), (2, 0), (2, 1), (2, 2), (2, 3)]


# ------------------------------------------------------------------ backward plans
def _bwd_desc(grad_caps=(100, 100, 80, 80), grad_tok=(512, 512, 256, 256), nbytes=(0, 0, 0, 0), **kw):
    bdesc = bd.ThdAttnBwdDesc()
    bdesc.fwd = _desc(**kw)
    for i in range(4):
        bdesc.cap_rows[i] = grad_caps[i]
        bdesc.stride_tok[i] = grad_tok[i]
        bdesc.stride_head[i] = 128
        bdesc.bytes[i] = nbytes[i]
    return bdesc


def _plan_bwd(bdesc):
    lib = bd.load_library()
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_attn_plan_bwd(ctypes.byref(h), ctypes.byref(bdesc), ctypes.byref(ws))
    kernel = lib.thd_attn_plan_kernel(h) if st == 0 else None
    if st == 0:
        lib.thd_attn_plan_destroy(h)
    return st, ws.value, kernel


def test_plan_bwd_validation_and_kernel_choice(lib):
    st, ws, kernel = _plan_bwd(_bwd_desc())
    assert st == 0 and ws % 256 == 0 and kernel == bd.KERNEL_TCGEN05
    # a gradient view with fewer rows than its primal view
    assert _plan_bwd(_bwd_desc(grad_caps=(100, 99, 80, 80)))[0] == 1
    # dQ allocation one element short of its all-axes span
    assert _plan_bwd(_bwd_desc(nbytes=(0, 100 * 512 * 2 - 2, 0, 0)))[0] == 4
    # forward checks still apply
    assert _plan_bwd(_bwd_desc(h_q=3, h_kv=2))[0] == 1
    assert _plan_bwd(_bwd_desc(dtype=torch.float32))[2] == bd.KERNEL_SIMT
    assert _plan_bwd(_bwd_desc(d=96, kernel=bd.KERNEL_TCGEN05))[0] == 2
    # a gradient token stride that is not a multiple of 16 bytes keeps the SIMT path
    assert _plan_bwd(_bwd_desc(grad_tok=(512, 516, 256, 256)))[2] == bd.KERNEL_SIMT


def test_fwd_rejects_backward_and_indexer_plans(lib):
    st, _, _ = _plan_bwd(_bwd_desc())
    assert st == 0
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.thd_attn_plan_bwd(ctypes.byref(h), ctypes.byref(_bwd_desc()), ctypes.byref(ws)) == 0
    args = [h] + [ctypes.c_void_p(256)] * 15 + [ctypes.c_void_p(0)]
    assert lib.thd_attn_fwd(*args) == 1
    lib.thd_attn_plan_destroy(h)


def test_static_entry_rejects_non_forward_plans_before_capacity(lib):
    """The workspace-free entry point refuses backward and indexer plans with
    THD_ERR_INVALID_ARG whatever their workspace size, and a forward plan larger than
    its static array with THD_ERR_WORKSPACE; all before any CUDA call."""
    cap = lib.thd_attn_static_workspace_capacity()
    out = ctypes.c_uint32()
    small_bwd = _bwd_desc()
    big_bwd = _bwd_desc()
    big_bwd.fwd.batch = cap // 32 + 1
    ix = _ix_desc()
    for make, desc in ((lib.thd_attn_plan_bwd, small_bwd), (lib.thd_attn_plan_bwd, big_bwd),
                       (lib.thd_indexer_plan, ix)):
        h = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        assert make(ctypes.byref(h), ctypes.byref(desc), ctypes.byref(ws)) == 0
        args = [h] + [ctypes.c_void_p(256)] * 14 + [ctypes.c_void_p(0)]
        assert lib.thd_attn_fwd_static_ws(*args) == 1
        assert lib.thd_attn_static_read_status(h, ctypes.byref(out), ctypes.c_void_p(0)) == 1
        lib.thd_attn_plan_destroy(h)
    big = bd.make_desc(torch.bfloat16, cap // 32 + 1, 1, 1, 64, (1, 1, 1, 1), (64, 64, 64, 64),
                       (64, 64, 64, 64), cap_rows_stats=1)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.thd_attn_plan(ctypes.byref(h), ctypes.byref(big), ctypes.byref(ws)) == 0
    assert ws.value > cap
    args = [h] + [ctypes.c_void_p(256)] * 14 + [ctypes.c_void_p(0)]
    assert lib.thd_attn_fwd_static_ws(*args) == 5
    lib.thd_attn_plan_destroy(h)


# ------------------------------------------------------------------- indexer plans
def _ix_desc(**kw):
    d = bd.ThdIndexerDesc()
    base = dict(dtype=0, batch=2, heads=64, d=128, topk=2048, cap_rows_q=8192, stride_tok_q=64 * 128,
                stride_head_q=128, cap_rows_k=131072, stride_tok_k=128, stride_tok_w=64, cap_rows_out=8192,
                max_seqlen_k=65536, kernel=bd.KERNEL_AUTO, flags=0)
    base.update(kw)
    for k_, v_ in base.items():
        setattr(d, k_, v_)
    return d


def _plan_ix(desc):
    lib = bd.load_library()
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_indexer_plan(ctypes.byref(h), ctypes.byref(desc), ctypes.byref(ws))
    kernel = lib.thd_attn_plan_kernel(h) if st == 0 else None
    if st == 0:
        lib.thd_attn_plan_destroy(h)
    return st, ws.value, kernel


def test_indexer_plan_validation_and_sizing(lib):
    st, ws, kernel = _plan_ix(_ix_desc())
    assert st == 0 and kernel == bd.KERNEL_TCGEN05
    # one float32 score row of max_seqlen_k (rounded to 128) per output row
    assert ws >= 8192 * 65536 * 4
    assert _plan_ix(_ix_desc(max_seqlen_k=1000))[1] < ws
    for kw in (dict(heads=0), dict(heads=129), dict(topk=0), dict(topk=4096), dict(d=0), dict(flags=1),
               dict(batch=-1), dict(dtype=2)):
        assert _plan_ix(_ix_desc(**kw))[0] == 1, kw
    assert _plan_ix(_ix_desc(heads=2))[2] == bd.KERNEL_SIMT          # H must be 4..64 for tensor cores
    assert _plan_ix(_ix_desc(heads=2, kernel=bd.KERNEL_TCGEN05))[0] == 2
    assert _plan_ix(_ix_desc(d=96))[2] == bd.KERNEL_SIMT


def test_indexer_key_schedule_sized_per_segment(lib):
    """Segments may share key rows (zigzag context-parallel chunks of one document),
    so the key-axis schedule holds batch x ceil(max_seqlen_k / 256) units (16 bytes
    each), not a bound derived from cap_rows_k: with the key and output capacities
    fixed, each extra segment adds at least 16 units of 256 keys at max_seqlen_k =
    4096."""
    small = dict(heads=8, d=64, topk=64, cap_rows_q=4096, stride_tok_q=8 * 64, stride_head_q=64,
                 cap_rows_k=4096, stride_tok_k=64, stride_tok_w=8, cap_rows_out=4096, max_seqlen_k=4096)
    sizes = [_plan_ix(_ix_desc(batch=b, **small)) for b in (1, 4, 16)]
    assert all(st == 0 and k == bd.KERNEL_TCGEN05 for st, _, k in sizes)
    ws = [w for _, w, _ in sizes]
    assert ws[1] - ws[0] >= 3 * 16 * 16 and ws[2] - ws[1] >= 12 * 16 * 16


def test_wrapper_plan_cache_is_bounded_lru(monkeypatch):
    """The one-call wrappers' plan cache keeps the most recently used plans only, so
    a caller whose shapes keep changing does not accumulate plans."""
    import collections
    monkeypatch.setattr(bd, "_PLAN_CACHE", collections.OrderedDict())
    made = []

    def make(i):
        return lambda: made.append(i) or ("plan", i)

    first = bd._cached_plan(("k", 0), make(0))
    for i in range(1, bd._PLAN_CACHE_SIZE):
        bd._cached_plan(("k", i), make(i))
    assert bd._cached_plan(("k", 0), make(-1)) is first          # hit: moved to the newest end
    bd._cached_plan(("k", "new"), make("new"))                    # evicts the oldest: key 1
    assert len(bd._PLAN_CACHE) == bd._PLAN_CACHE_SIZE
    assert ("k", 1) not in bd._PLAN_CACHE and ("k", 0) in bd._PLAN_CACHE
    assert -1 not in made


def test_plan_builders_reject_mixed_storage_types(lib):
    """One descriptor dtype covers every tensor of a plan: mixed storage types are
    a caller error, refused before any plan exists."""
    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(8, 2, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        bd.plan_for_tensors(q, k, q, q, 1, 8, bd.STATS_TOKEN_MAJOR)
    with pytest.raises(ValueError):
        bd.plan_bwd_for_tensors(q, q, q, q, q, q, k, q, 1, 8, bd.STATS_TOKEN_MAJOR)
    w = torch.zeros(8, 2, dtype=torch.float32)
    idx = torch.zeros(8, 4, dtype=torch.int32)
    with pytest.raises(ValueError):
        bd.indexer_plan_for_tensors(q, torch.zeros(8, 64, dtype=torch.float16), w, idx, 1, 4)
    assert bd.plan_for_tensors(q, q, q, q, 1, 8, bd.STATS_TOKEN_MAJOR).workspace_bytes > 0
