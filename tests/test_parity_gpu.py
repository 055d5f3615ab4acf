"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from ragged_varlen_attention_gb300 import binding as bd
from ragged_varlen_attention_gb300 import workloads as wl
from tests import schedule_mirror
from tests.gpu_harness import TOL, check_parity, check_untouched, run_thd
from tests.helpers import max_abs_finite

pytestmark = pytest.mark.gpu

KERNELS = [bd.KERNEL_AUTO, bd.KERNEL_SIMT]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from ragged_varlen_attention_gb300 import build
    build.build()
    bd.load_library()


# scaled-down variants of the named workloads: same generators and structure,
# sizes the oracle finishes in seconds while still spanning several tiles and
# ragged tails
SMALL = {
    "tiny_padded": {},
    "padded_causal": dict(b=4, h=4, min_len=64, max_len=400),
    "mixed_gqa": dict(b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2),
    "separate_padding": dict(b=6, max_len=500, h=4),
    "cp_chunks": dict(docs=2, k_len=2048, q_len=384, h=2),   # 16 KV tiles: the key range splits
}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_workload_parity_small(name, kernel):
    batch = wl.make(name, **SMALL[name])
    res = run_thd(batch, kernel=kernel)
    assert res["status"] == 0
    check_parity(batch, res)
    check_untouched(batch, res)


def _sample_rows(batch, seed=0, per_seq=512):
    """``per_seq`` rows of every sequence (all rows of shorter ones): the tile and
    sub-tile boundaries and the ragged tail, the rest in runs of 64 consecutive rows
    at random positions."""
    rng = np.random.default_rng(seed)
    out = {}
    for b, L in enumerate(batch.lens_q()):
        L = int(L)
        if L <= per_seq:
            out[b] = list(range(L))
            continue
        rows = {r for r in (0, 1, 127, 128, 129, 255, 256, 257, 383, 384, 511, 512, L - 129, L - 128, L - 2, L - 1)
                if 0 <= r < L}
        free = np.setdiff1d(np.arange(L), np.array(sorted(rows)))
        while len(rows) < per_seq:
            # a run of up to 64 rows starting at a row not taken yet
            r0 = int(rng.choice(free))
            run = range(r0, min(L, r0 + 64, r0 + per_seq - len(rows)))
            rows.update(run)
            free = free[(free < run.start) | (free >= run.stop)]
        out[b] = sorted(rows)
    return out


# full-size workloads in the benchmark's launch configuration (KV split on where the
# plan allows it), every row of every head against the oracle (the 128k-token
# context-parallel chunks are ~4.4 TFLOP of float64 work for the oracle)
@pytest.mark.parametrize("name", ["padded_causal", "mixed_gqa", "separate_padding", "cp_chunks"])
def test_workload_full_size(name):
    """O and LSE of the full-size workloads against the oracle, element by element on
    every row and head; every other byte of O and Stats untouched."""
    batch = wl.make(name)
    res = run_thd(batch)
    assert res["status"] == 0
    check_parity(batch, res)
    check_untouched(batch, res)


@pytest.mark.parametrize("name", ["cp_chunks", "separate_padding", "mixed_gqa"])
@pytest.mark.parametrize("k", [1, 2])
def test_workload_full_size_other_seeds(name, k):
    """Two more seeds of each workload at full size: 512 rows of every sequence (for
    every head) against the oracle -- rows are independent, so a subset is exact --
    and every other byte of O and Stats untouched."""
    batch = wl.make(name, seed=wl.WORKLOAD_SEEDS[name] * 100 + k)
    res = run_thd(batch)
    assert res["status"] == 0
    check_parity(batch, res, row_subset=_sample_rows(batch, seed=k))
    check_untouched(batch, res)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("seed", range(12))
def test_random_packs(seed, kernel):
    rng = np.random.default_rng(1000 + seed)
    dtype = ["bf16", "fp16", "fp32"][seed % 3]
    d = [64, 128, 32, 16][seed % 4] if dtype != "fp32" else [16, 64, 128][seed % 3]
    h_kv = int(rng.integers(1, 4))
    h_q = h_kv * int(rng.integers(1, 4))
    batch = wl.random_pack(2000 + seed, batch=int(rng.integers(1, 7)), max_len=int(rng.integers(1, 700)),
                           h_q=h_q, h_kv=h_kv, d=d, dtype=dtype)
    gaps = tuple(int(x) for x in rng.integers(0, 4, size=4))
    res = run_thd(batch, kernel=kernel, gaps=gaps)
    assert res["status"] == 0
    check_parity(batch, res)
    check_untouched(batch, res)


@pytest.mark.parametrize("seed", [2600, 2603, 2602])
def test_split_ragged_packs(seed):
    """Few long ragged sequences (under four waves of units, so pairs of 16 or more
    KV tiles are processed as two halves and merged): partial tiles, mixed masks,
    causal offsets and both Stats layouts through the split and combine path."""
    d, dtype = {2600: (128, "bf16"), 2603: (64, "fp16"), 2602: (128, "bf16")}[seed]
    batch = wl.random_pack(seed, batch=3, max_len=3000, h_q=2, h_kv=1, d=d, dtype=dtype, allow_empty=False)
    res = run_thd(batch)
    hdr, _, _, _ = res["plan"].workspace_layout
    n_split = int(res["ws"].cpu().numpy()[hdr:hdr + 128].view(np.uint32)[16])
    assert res["status"] == 0
    assert n_split > 0, "no pair was split"
    check_parity(batch, res)
    check_untouched(batch, res)


def test_tail_split_parts():
    """Long-context chunks whose halved key ranges leave a partial last wave: the
    cheapest pairs are processed in eight parts (checked in the tile list) and merged
    by the combine kernel; sampled rows against the oracle, every row against the
    unsplit path, and no other byte of O and Stats touched."""
    batch = wl.make("cp_chunks", **TAIL_CASE)
    res = run_thd(batch)
    assert res["status"] == 0
    hdr, _, _, pairs_off = res["plan"].workspace_layout
    ws = res["ws"].cpu().numpy()
    n_entries = int(ws[hdr:hdr + 128].view(np.uint32)[2])
    parts = ws[pairs_off:pairs_off + 16 * n_entries].view(np.int32).reshape(n_entries, 4)[:, 2] & 0xFF
    assert (parts == 8).sum() > 0 and (parts == 2).sum() > 0
    check_parity(batch, res, row_subset=_sample_rows(batch, seed=7))
    check_untouched(batch, res)
    ref = run_thd(batch, flags=bd.FLAG_NO_KV_SPLIT)
    assert ref["status"] == 0
    assert max_abs_finite(res["o"].float().numpy(), ref["o"].float().numpy()) <= 2e-2
    assert max_abs_finite(res["stats"].numpy(), ref["stats"].numpy()) <= 1e-3


@pytest.mark.parametrize("kernel", KERNELS)
def test_kv_interleaved_view_equals_contiguous(kernel):
    """K/V as views of an interleaved [T, 2, H, D] buffer (token stride 2*H*D) give
    the same bits as contiguous copies (cudnn-frontend PR #516 layout)."""
    batch = wl.random_pack(77, batch=4, max_len=300, h_q=4, h_kv=4, d=128, dtype="bf16")
    a = run_thd(batch, kernel=kernel)
    b = run_thd(batch, kernel=kernel, gaps=(0, 1, 1, 0))
    assert torch.equal(a["o"].view(torch.int16), b["o"].view(torch.int16))
    assert torch.equal(a["stats"].view(torch.int32), b["stats"].view(torch.int32))


TAIL_CASE = dict(docs=2, k_len=16384, q_len=1536, h=16)

SCHEDULE_CASES = [
    ("mixed_gqa", {}, bd.KERNEL_AUTO, 0),                      # many units: no split
    ("mixed_gqa", {}, bd.KERNEL_SIMT, 0),
    ("cp_chunks", dict(docs=2, k_len=2048, q_len=768, h=4), bd.KERNEL_AUTO, 0),   # split
    ("cp_chunks", dict(docs=2, k_len=2048, q_len=768, h=4), bd.KERNEL_AUTO, bd.FLAG_NO_KV_SPLIT),
    # 12 pairs of ~128 tiles, 16 heads: halves give 2.5 waves, the last wave's pairs in 8 parts
    ("cp_chunks", TAIL_CASE, bd.KERNEL_AUTO, 0),
]


@pytest.mark.parametrize("name,kw,kernel,flags", SCHEDULE_CASES)
def test_schedule_matches_cpu_mirror(name, kw, kernel, flags):
    batch = wl.make(name, **kw)
    res = run_thd(batch, kernel=kernel, flags=flags)
    plan = res["plan"]
    ws = res["ws"].cpu().numpy()
    hdr, meta_off, base_off, pairs_off = plan.workspace_layout
    header = ws[hdr:hdr + 128].view(np.uint32)
    meta_exp, pairs_exp, status_exp, n_base = schedule_mirror.mirror(
        batch, plan.rows_per_unit, plan.keys_per_tile, plan.max_pairs)
    num_ctas = min(torch.cuda.get_device_properties(0).multi_processor_count, 2 * plan.max_pairs * batch.h_q)
    allow = plan.kernel == bd.KERNEL_TCGEN05 and not flags
    max_split = min(plan.max_pairs, -(-4 * 160 // batch.h_q)) if allow else 0
    entries, n_split = schedule_mirror.split_entries(pairs_exp, batch.h_q, num_ctas, max_split, allow)
    n_exp = len(entries)
    assert header[1] == status_exp and header[2] == n_exp and header[3] == n_exp * batch.h_q
    assert header[16] == n_split
    starts = schedule_mirror.group_starts([(b, r, c) for b, r, _, _, c in entries])
    assert list(header[4:4 + len(starts)]) == starts
    meta = ws[meta_off:meta_off + 48 * batch.batch].view(np.int32).reshape(batch.batch, 12)
    assert np.array_equal(meta, meta_exp)
    recs = ws[pairs_off:pairs_off + 16 * n_exp].view(np.int32).reshape(n_exp, 4)
    # same multiset of (b, row0, part, parts); costs non-increasing along the list;
    # part i of a split pair has partial slot slot0 + i, and the slots of all split
    # pairs are 0 .. (their parts) - 1
    cost = {(b, r, i, n): c for b, r, i, n, c in entries}
    got = [(int(x[0]), int(x[1]), int(x[2]) >> 8, int(x[2]) & 0xFF) for x in recs]
    assert sorted(got) == sorted(cost)
    costs = [cost[g] for g in got]
    assert all(x >= y for x, y in zip(costs, costs[1:]))
    slots = {}
    for g, x in zip(got, recs):
        if g[3] > 1:
            slots.setdefault((g[0], g[1]), {})[g[2]] = int(x[3])
        else:
            assert int(x[3]) == -1
    assert len(slots) == n_split
    for d in slots.values():
        assert d == {i: d[0] + i for i in range(len(d))}
    assert sorted(v for d in slots.values() for v in d.values()) == list(range(sum(len(d) for d in slots.values())))


@pytest.mark.parametrize("name", ["cp_chunks", "mixed_gqa", "separate_padding"])
def test_kv_split_matches_unsplit(name):
    """The split path (two halves of each key range merged by log-sum-exp weights)
    agrees with the unsplit path and with the oracle."""
    batch = wl.make(name, **SMALL[name])
    a = run_thd(batch)
    b = run_thd(batch, flags=bd.FLAG_NO_KV_SPLIT)
    assert a["status"] == 0 and b["status"] == 0
    check_parity(batch, a)
    check_parity(batch, b)
    check_untouched(batch, a)
    tol_o, tol_l = TOL[batch.dtype]
    diff = torch.nan_to_num((a["o"].float() - b["o"].float()).abs(), nan=0.0)
    assert float(diff.max()) <= tol_o


@pytest.mark.parametrize("kernel", KERNELS)
def test_deterministic(kernel):
    batch = wl.padded_causal()
    a = run_thd(batch, kernel=kernel)
    b = run_thd(batch, kernel=kernel, reps=3)
    assert torch.equal(a["o"].view(torch.int16), b["o"].view(torch.int16))
    assert torch.equal(a["stats"].view(torch.int32), b["stats"].view(torch.int32))


def test_invalid_sequences_flagged_and_untouched():
    batch = wl.random_pack(5, batch=5, max_len=100, h_q=2, h_kv=2, d=64, dtype="bf16",
                           allow_empty=False)
    batch.off_k = batch.off_k.copy()
    batch.off_k[1] = batch.k.shape[0]                 # K rows past capacity
    batch.mask_type = batch.mask_type.copy()
    batch.mask_type[3] = 7                            # unknown mask
    res = run_thd(batch)
    assert res["status"] == bd.DEV_BAD_OFFSET | bd.DEV_BAD_MASK
    # the valid sequences are still right; the invalid ones left their rows alone
    good = wl.ThdBatch(**{**batch.__dict__})
    good.cu_seqlens_q = batch.cu_seqlens_q.copy()
    lens = batch.lens_q()
    lens[[1, 3]] = 0
    good.cu_seqlens_q = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    lk = batch.lens_k()
    lk[[1, 3]] = 0
    good.cu_seqlens_kv = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    good.mask_type[3] = 0
    check_parity(good, res)
    check_untouched(good, res)


def test_cuda_graph_replay():
    batch = wl.mixed_gqa()
    ref = run_thd(batch)
    dev = ref["dev"]
    plan = ref["plan"]
    ws = torch.empty_like(ref["ws"])
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        bd.thd_attn_fwd(plan, dev["q"], dev["k"], dev["v"], dev["o"], dev["stats"], dev["cu_q"],
                        dev["cu_k"], *dev["offs"], dev["mask"], dev["qco"], ws, s)
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        bd.thd_attn_fwd(plan, dev["q"], dev["k"], dev["v"], dev["o"], dev["stats"], dev["cu_q"],
                        dev["cu_k"], *dev["offs"], dev["mask"], dev["qco"], ws, s)
    dev["o"].zero_()
    dev["stats"].zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check_parity(batch, dict(o=dev["o"].cpu(), stats=dev["stats"].cpu()))


def test_empty_batch_and_all_empty_sequences():
    batch = wl.random_pack(9, batch=3, max_len=0, h_q=2, h_kv=1, d=64, dtype="fp16")
    res = run_thd(batch)
    assert res["status"] == 0
    check_untouched(batch, res)


def test_bounded_wait_gives_up_and_context_survives():
    """A wait that nothing completes (test hook) ends in ~100 ms: the kernel sets the
    timeout bit, drains and returns; the next call on the same context is correct."""
    import time
    batch = wl.make("cp_chunks", **SMALL["cp_chunks"])
    t0 = time.time()
    res = run_thd(batch, flags=bd.FLAG_TEST_STALL)
    assert time.time() - t0 < 30
    assert res["status"] & bd.DEV_WAIT_TIMEOUT
    good = run_thd(batch)
    assert good["status"] == 0
    check_parity(batch, good)
    check_untouched(batch, good)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("mult", [0, 2, 4])
def test_element_offsets_equal_row_offsets(kernel, mult):
    """Offsets in element units (row x token stride, optionally divided by a
    multiplier that the device applies back) give the same bits as row offsets,
    with per-tensor token-stride gaps. Token-major Stats (token stride h_q = 4) keep
    every element offset divisible by the multiplier."""
    batch = wl.random_pack(300 + mult, batch=5, max_len=300, h_q=4, h_kv=2, d=64, dtype="bf16",
                           stats_layout=wl.STATS_TOKEN_MAJOR)
    gaps = (1, 2, 0, 3)
    a = run_thd(batch, kernel=kernel, gaps=gaps)
    b = run_thd(batch, kernel=kernel, gaps=gaps, element_mult=mult)
    assert a["status"] == 0 and b["status"] == 0
    assert torch.equal(a["o_backing"].view(torch.int16), b["o_backing"].view(torch.int16))
    assert torch.equal(a["stats"].view(torch.int32), b["stats"].view(torch.int32))
    check_parity(batch, b)


def test_element_offset_not_a_whole_row_is_flagged():
    batch = wl.random_pack(321, batch=3, max_len=100, h_q=2, h_kv=2, d=64, dtype="bf16", allow_empty=False)
    res = run_thd(batch, element_mult=1)
    assert res["status"] == 0
    # shift sequence 1's K offset by one element: no longer a whole row
    dev = res["dev"]
    offs = [t.clone() for t in dev["offs"]]
    offs[1][1] += 1
    o = torch.empty_like(dev["o"])
    o.view(torch.uint8).fill_(wl.SENTINEL_BYTE)
    plan = res["plan"]
    bd.thd_attn_fwd(plan, dev["q"], dev["k"], dev["v"], o, dev["stats"], dev["cu_q"], dev["cu_k"], *offs,
                    dev["mask"], dev["qco"], res["ws"])
    assert bd.thd_attn_read_status(plan, res["ws"]) == bd.DEV_BAD_OFFSET
    # sequence 1's rows untouched, the others written
    o1 = o.cpu().view(torch.uint8)[int(batch.off_o[1]):int(batch.off_o[1]) + int(batch.lens_q()[1])]
    assert (o1 == wl.SENTINEL_BYTE).all()


# ------------------------------------------------------------------ left window
def _with_window(batch: wl.ThdBatch, windows) -> wl.ThdBatch:
    import dataclasses
    w = np.array([windows[i % len(windows)] for i in range(batch.batch)], dtype=np.int32)
    return dataclasses.replace(batch, window_left=w)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("seed", range(8))
def test_random_packs_window(seed, kernel):
    """Per-sequence left windows on the causal masks (TransformerEngine PR #3274,
    per-policy windows): zero, short, longer than the sequence and unbounded, over
    random ragged packs with mixed masks and causal offsets."""
    rng = np.random.default_rng(3000 + seed)
    dtype = ["bf16", "fp16"][seed % 2]
    d = [64, 128][(seed // 2) % 2]
    h_kv = int(rng.integers(1, 3))
    h_q = h_kv * int(rng.integers(1, 3))
    batch = wl.random_pack(4000 + seed, batch=int(rng.integers(1, 7)), max_len=int(rng.integers(1, 900)),
                           h_q=h_q, h_kv=h_kv, d=d, dtype=dtype, with_window=True)
    res = run_thd(batch, kernel=kernel)
    assert res["status"] == 0
    check_parity(batch, res)
    check_untouched(batch, res)


@pytest.mark.parametrize("windows", [(0,), (1, 127, 128, 129), (300, 700), (-1, 5000)])
def test_window_split_matches_unsplit(windows):
    """Window ranges through the KV split (halves of the pair's tile span) agree
    with the unsplit path and with the oracle."""
    batch = _with_window(wl.make("cp_chunks", **SMALL["cp_chunks"]), windows)
    a = run_thd(batch)
    b = run_thd(batch, flags=bd.FLAG_NO_KV_SPLIT)
    assert a["status"] == 0 and b["status"] == 0
    check_parity(batch, a)
    check_parity(batch, b)
    check_untouched(batch, a)


@pytest.mark.parametrize("kernel", KERNELS)
def test_window_long_sequences(kernel):
    """Windows far shorter than the sequence: most KV tiles of each unit are
    skipped, and the two query sub-tiles of a unit start on different tiles."""
    batch = _with_window(wl.padded_causal(b=3, h=2, min_len=2500, max_len=3000), (256, 1000, 70))
    res = run_thd(batch, kernel=kernel)
    assert res["status"] == 0
    check_parity(batch, res)
    check_untouched(batch, res)


def test_window_schedule_matches_cpu_mirror():
    """With a window the pair cost is the span from the first row's lowest visible
    tile to the last row's highest; setup metadata and order match the CPU mirror."""
    batch = _with_window(wl.make("cp_chunks", docs=2, k_len=2048, q_len=768, h=4), (200, -1, 600, 0))
    res = run_thd(batch)
    plan = res["plan"]
    ws = res["ws"].cpu().numpy()
    hdr, meta_off, base_off, pairs_off = plan.workspace_layout
    header = ws[hdr:hdr + 128].view(np.uint32)
    meta_exp, pairs_exp, status_exp, _ = schedule_mirror.mirror(
        batch, plan.rows_per_unit, plan.keys_per_tile, plan.max_pairs)
    meta = ws[meta_off:meta_off + 48 * batch.batch].view(np.int32).reshape(batch.batch, 12)
    assert np.array_equal(meta, meta_exp)
    num_ctas = min(torch.cuda.get_device_properties(0).multi_processor_count, 2 * plan.max_pairs * batch.h_q)
    max_split = min(plan.max_pairs, -(-4 * 160 // batch.h_q))
    entries, n_split = schedule_mirror.split_entries(pairs_exp, batch.h_q, num_ctas, max_split, True)
    assert header[1] == status_exp and header[2] == len(entries) and header[16] == n_split
    starts = schedule_mirror.group_starts([(b, r, c) for b, r, _, _, c in entries])
    assert list(header[4:4 + len(starts)]) == starts
    check_parity(batch, res)
