"""The FLOP and byte counts bench.py reports, checked on the CPU against
independent counts: the oracle's visible-entry count for attention (with and
without windows) and brute-force enumeration for the indexer's visible pairs."""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import bench
from oracle import unmasked_entries
from ragged_varlen_attention_gb300 import workloads as wl

SMALL = {
    "tiny_padded": {},
    "padded_causal": dict(b=4, h=4, min_len=64, max_len=400),
    "mixed_gqa": dict(b=6, median=128, max_len=700, total=1900, h_q=8, h_kv=2),
    "separate_padding": dict(b=6, max_len=500, h=4),
    "cp_chunks": dict(docs=2, k_len=1024, q_len=384, h=2),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("window", [None, 0, 37, 300])
def test_attention_flop_count_matches_oracle(name, window):
    batch = wl.make(name, **SMALL[name])
    if window is not None:
        batch = dataclasses.replace(batch, window_left=np.full(batch.batch, window, dtype=np.int32))
    got = bench.unmasked_entries(batch)
    want = unmasked_entries(batch.cu_seqlens_q, batch.cu_seqlens_kv, batch.mask_type, batch.q_causal_offset,
                            batch.h_q, window_left=batch.window_left)
    assert got == want


def test_full_size_cp_chunks_count():
    # 2 docs x sum_{i<4096} (61440 + i + 1) visible keys x 16 heads
    per_doc = sum(61440 + i + 1 for i in range(4096))
    batch = wl.make("cp_chunks")
    assert bench.unmasked_entries(batch) == 2 * 16 * per_doc == 8_321_564_672


@pytest.mark.parametrize("seed", range(4))
def test_indexer_visible_pairs_brute_force(seed):
    b = wl.indexer_random_pack(9000 + seed, batch=4, max_len=60, heads=2, d=16, topk=4)
    want = 0
    for s in range(b.batch):
        lq, lk = int(b.lens_q()[s]), int(b.lens_k()[s])
        mt = int(b.mask_type[s])
        c = None if mt == 0 else (0 if mt == 1 else int(b.q_causal_offset[s]))
        for i in range(lq):
            for j in range(lk):
                want += 1 if (c is None or j <= i + c) else 0
    assert bench.indexer_visible_pairs(b) == want


def test_valid_bytes_counts_each_valid_row_once():
    batch = wl.make("padded_causal", **SMALL["padded_causal"])
    e = 2
    tq, tk = int(batch.lens_q().sum()), int(batch.lens_k().sum())
    assert bench.valid_bytes(batch) == (2 * tq * batch.h_q * batch.d + 2 * tk * batch.h_kv * batch.d) * e \
        + 4 * tq * batch.h_q
