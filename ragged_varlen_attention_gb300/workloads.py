"""Seeded synthetic packed-THD batches.

This module only draws inputs: sequence lengths, gap sizes, mask choices and
N(0, 1) tensor values, and lays them out in rows. It holds none of the
attention arithmetic, so both the CUDA path's tests/bench and the CPU oracle
can consume the same batch.

Named workloads (shapes follow the pages' packed-THD examples):

* ``tiny_padded``      -- 3 sequences, lengths [3, 2, 4] with one identifier row after
  each (cu_seqlens [0,3,5,9], cu_seqlens_padded [0,4,8,13]), h=2, d=16, fp32,
  masks [causal, none, causal], token-major LSE.
* ``padded_causal``    -- 8 sequences, lengths U{64..1024}, 0-16 pad rows after
  each, h=16, d=128, bf16, top-left causal, head-major LSE.
* ``mixed_gqa``        -- 32 sequences, lognormal lengths (median 512, clipped to
  [16, 4096], ~32k tokens), 0-8 pad rows, h_q=32/h_kv=8, d=128, bf16, causal flag
  ~ Bernoulli(0.5), token-major LSE.
* ``cp_chunks``        -- 2 documents of 65536 keys, a 4096-row query chunk each at
  causal offset k_len - q_len (bottom-right causal), h=16, d=128, bf16, head-major
  LSE.
* ``separate_padding`` -- 64 sequences, lengths U{0..4096} (one forced to 0), Q/O
  rows padded to multiples of 64 with NaN, K/V packed with 1-row identifier gaps,
  h=32, d=64, fp16, masks drawn from {none, causal, bottom-right causal},
  token-major LSE.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

MASK_NONE, MASK_TOP_LEFT, MASK_BOTTOM_RIGHT = 0, 1, 2
STATS_TOKEN_MAJOR, STATS_HEAD_MAJOR = 0, 1

# byte pattern pre-filled into every output buffer; rows the kernel must not
# touch are compared against it bit for bit
SENTINEL_BYTE = 0xA5

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}

WORKLOAD_SEEDS = {"tiny_padded": 101, "padded_causal": 102, "mixed_gqa": 103, "zigzag_chunks": 108,
                  "cp_chunks": 104, "separate_padding": 105, "cp_chunks_one_doc": 104}


@dataclass
class ThdBatch:
    """One packed-THD problem: metadata (host numpy) and tensors (host torch)."""
    name: str
    dtype: str
    h_q: int
    h_kv: int
    d: int
    cu_seqlens_q: np.ndarray      # int32 [B+1]
    cu_seqlens_kv: np.ndarray     # int32 [B+1]
    off_q: np.ndarray             # int32 [B+1] row offsets (entry B = end marker)
    off_k: np.ndarray
    off_v: np.ndarray
    off_o: np.ndarray
    off_s: np.ndarray
    mask_type: np.ndarray         # int8 [B]
    q_causal_offset: np.ndarray | None  # int32 [B] or None
    stats_layout: int
    q: torch.Tensor               # [cap_q, h_q, d] storage dtype
    k: torch.Tensor               # [cap_k, h_kv, d]
    v: torch.Tensor               # [cap_v, h_kv, d]
    cap_o: int
    cap_s: int
    softmax_scale: float | None = None
    window_left: np.ndarray | None = None   # int32 [B] or None
    notes: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens_q) - 1

    @property
    def torch_dtype(self):
        return _TORCH_DTYPE[self.dtype]

    @property
    def stats_strides(self):
        """(token stride, head stride) of the flat Stats buffer, in elements."""
        if self.stats_layout == STATS_TOKEN_MAJOR:
            return self.h_q, 1
        return 1, self.cap_s

    @property
    def stats_numel(self) -> int:
        return self.cap_s * self.h_q

    def lens_q(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q.astype(np.int64))

    def lens_k(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_kv.astype(np.int64))

    def o_init(self) -> torch.Tensor:
        """Output buffer pre-filled with the sentinel byte pattern."""
        t = torch.empty((self.cap_o, self.h_q, self.d), dtype=self.torch_dtype)
        t.view(torch.uint8).fill_(SENTINEL_BYTE)
        return t

    def stats_init(self) -> torch.Tensor:
        t = torch.empty((self.stats_numel,), dtype=torch.float32)
        t.view(torch.uint8).fill_(SENTINEL_BYTE)
        return t


def _normal(rng: np.random.Generator, shape, dtype: str) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(_TORCH_DTYPE[dtype])


def _fill_rows(t: torch.Tensor, rows: np.ndarray, value: float) -> None:
    if len(rows):
        t[torch.from_numpy(rows.astype(np.int64))] = value


def _pad_rows(cap: int, starts: np.ndarray, lens: np.ndarray) -> np.ndarray:
    """Rows of [0, cap) not covered by any [start, start+len)."""
    used = np.zeros(cap, dtype=bool)
    for s, n in zip(starts, lens):
        used[s:s + n] = True
    return np.nonzero(~used)[0]


def _cumsum0(x) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(x, dtype=np.int64))]).astype(np.int32)


def tiny_padded(seed: int = WORKLOAD_SEEDS["tiny_padded"]) -> ThdBatch:
    rng = np.random.default_rng(seed)
    cu = np.array([0, 3, 5, 9], dtype=np.int32)
    padded = np.array([0, 4, 8, 13], dtype=np.int32)
    cap, h, d = 13, 2, 16
    q, k, v = (_normal(rng, (cap, h, d), "fp32") for _ in range(3))  # identifier rows: N(0,1)
    return ThdBatch("tiny_padded", "fp32", h, h, d, cu, cu.copy(), padded, padded.copy(),
                    padded.copy(), padded.copy(), padded.copy(),
                    np.array([MASK_TOP_LEFT, MASK_NONE, MASK_TOP_LEFT], dtype=np.int8), None,
                    STATS_TOKEN_MAJOR, q, k, v, cap, cap)


def padded_causal(seed: int = WORKLOAD_SEEDS["padded_causal"], b: int = 8, h: int = 16, d: int = 128,
                  min_len: int = 64, max_len: int = 1024) -> ThdBatch:
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len, size=b, endpoint=True)
    gaps = rng.integers(0, 16, size=b, endpoint=True)
    cu = _cumsum0(lens)
    padded = _cumsum0(lens + gaps)
    cap = int(padded[-1])
    q, k, v = (_normal(rng, (cap, h, d), "bf16") for _ in range(3))
    pads = _pad_rows(cap, padded[:-1], lens)
    for t in (q, k, v):
        _fill_rows(t, pads, float("nan"))
    return ThdBatch("padded_causal", "bf16", h, h, d, cu, cu.copy(), padded, padded.copy(),
                    padded.copy(), padded.copy(), padded.copy(),
                    np.full(b, MASK_TOP_LEFT, dtype=np.int8), None, STATS_HEAD_MAJOR,
                    q, k, v, cap, cap)


def mixed_gqa(seed: int = WORKLOAD_SEEDS["mixed_gqa"], sigma: float = 1.35, b: int = 32,
              median: int = 512, max_len: int = 4096, total: int = 32768, h_q: int = 32,
              h_kv: int = 8, d: int = 128) -> ThdBatch:
    rng = np.random.default_rng(seed)
    while True:
        lens = np.clip(np.round(median * np.exp(sigma * rng.standard_normal(b))), 16, max_len)
        lens = lens.astype(np.int64)
        if abs(int(lens.sum()) - total) <= total // 10:
            break
    gaps = rng.integers(0, 8, size=b, endpoint=True)
    cu = _cumsum0(lens)
    padded = _cumsum0(lens + gaps)
    cap = int(padded[-1])
    q = _normal(rng, (cap, h_q, d), "bf16")
    k = _normal(rng, (cap, h_kv, d), "bf16")
    v = _normal(rng, (cap, h_kv, d), "bf16")
    pads = _pad_rows(cap, padded[:-1], lens)
    for t in (q, k, v):
        _fill_rows(t, pads, float("nan"))
    mask = rng.integers(0, 2, size=b).astype(np.int8)   # Bernoulli(0.5): 0 none, 1 causal
    return ThdBatch("mixed_gqa", "bf16", h_q, h_kv, d, cu, cu.copy(), padded, padded.copy(),
                    padded.copy(), padded.copy(), padded.copy(), mask, None, STATS_TOKEN_MAJOR,
                    q, k, v, cap, cap)


def cp_chunks(seed: int = WORKLOAD_SEEDS["cp_chunks"], docs: int = 2, k_len: int = 65536,
              q_len: int = 4096, h: int = 16, d: int = 128) -> ThdBatch:
    rng = np.random.default_rng(seed)
    cu_k = _cumsum0([k_len] * docs)
    cu_q = _cumsum0([q_len] * docs)
    q = _normal(rng, (docs * q_len, h, d), "bf16")
    k = _normal(rng, (docs * k_len, h, d), "bf16")
    v = _normal(rng, (docs * k_len, h, d), "bf16")
    qco = np.full(docs, k_len - q_len, dtype=np.int32)
    return ThdBatch("cp_chunks", "bf16", h, h, d, cu_q, cu_k, cu_q.copy(), cu_k.copy(),
                    cu_k.copy(), cu_q.copy(), cu_q.copy(),
                    np.full(docs, MASK_BOTTOM_RIGHT, dtype=np.int8), qco, STATS_HEAD_MAJOR,
                    q, k, v, docs * q_len, docs * q_len)


def separate_padding(seed: int = WORKLOAD_SEEDS["separate_padding"], b: int = 64,
                     max_len: int = 4096, h: int = 32, d: int = 64, q_multiple: int = 64) -> ThdBatch:
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_len, size=b, endpoint=True)
    lens[int(rng.integers(0, b))] = 0
    cu = _cumsum0(lens)
    q_slots = (lens + q_multiple - 1) // q_multiple * q_multiple
    off_q = _cumsum0(q_slots)
    off_k = _cumsum0(lens + 1)            # one identifier row after each sequence
    cap_q, cap_k = int(off_q[-1]), int(off_k[-1])
    q = _normal(rng, (cap_q, h, d), "fp16")
    k = _normal(rng, (cap_k, h, d), "fp16")
    v = _normal(rng, (cap_k, h, d), "fp16")
    _fill_rows(q, _pad_rows(cap_q, off_q[:-1], lens), float("nan"))
    mask = rng.integers(0, 3, size=b).astype(np.int8)
    return ThdBatch("separate_padding", "fp16", h, h, d, cu, cu.copy(), off_q, off_k,
                    off_k.copy(), off_q.copy(), off_q.copy(), mask, None, STATS_TOKEN_MAJOR,
                    q, k, v, cap_q, cap_q)


def zigzag_chunks(seed: int = WORKLOAD_SEEDS["zigzag_chunks"], docs: int = 2, doc_len: int = 4096, cp_size: int = 2, ranks=(0, 1),
                  h_q: int = 4, h_kv: int = 2, d: int = 128, dtype: str = "bf16",
                  stats_layout: int = STATS_TOKEN_MAJOR) -> ThdBatch:
    """Zigzag context-parallel query chunks as attention segments (Megatron-LM PR
    #14, the packed-CP paths): each document is cut into 2 * cp_size chunks of
    doc_len / (2 * cp_size) rows and rank r holds chunks r and 2 * cp_size - 1 - r.
    Every chunk is one THD segment whose queries see the key prefix ending with the
    chunk, bottom-right aligned at q_causal_offset = the chunk's first row in the
    document. The segments of one document read the SAME K/V rows (equal off_k and
    off_v, adjacent in the batch), so their key ranges overlap and their dK / dV
    add up; documents have K/V rows of their own."""
    rng = np.random.default_rng(seed)
    c = doc_len // (2 * cp_size)
    chunks = [ch for r in ranks for ch in (r, 2 * cp_size - 1 - r)]
    lq = np.full(docs * len(chunks), c, dtype=np.int64)
    lk = np.array([(ch + 1) * c for _ in range(docs) for ch in chunks], dtype=np.int64)
    off_q = _cumsum0(lq)
    off_k = np.repeat(np.arange(docs, dtype=np.int64) * doc_len, len(chunks)).astype(np.int32)
    off_k = np.concatenate([off_k, [docs * doc_len]]).astype(np.int32)
    cap_q = int(lq.sum())
    q = _normal(rng, (cap_q, h_q, d), dtype)
    k = _normal(rng, (docs * doc_len, h_kv, d), dtype)
    v = _normal(rng, (docs * doc_len, h_kv, d), dtype)
    qco = np.array([ch * c for _ in range(docs) for ch in chunks], dtype=np.int32)
    return ThdBatch("zigzag_chunks", dtype, h_q, h_kv, d, _cumsum0(lq), _cumsum0(lk), off_q, off_k,
                    off_k.copy(), off_q.copy(), off_q.copy(),
                    np.full(len(lq), MASK_BOTTOM_RIGHT, dtype=np.int8), qco, stats_layout, q, k, v, cap_q, cap_q)


def cp_chunks_one_doc(seed: int = WORKLOAD_SEEDS["cp_chunks"], **kw) -> ThdBatch:
    """One document of the cp_chunks workload (65536 keys, a 4096-row chunk): the same
    per-unit work on half the units, for profiler captures that must stay small."""
    return cp_chunks(seed=seed, docs=1, **kw)


WORKLOADS = {"tiny_padded": tiny_padded, "padded_causal": padded_causal,
             "mixed_gqa": mixed_gqa, "cp_chunks": cp_chunks,
             "separate_padding": separate_padding, "zigzag_chunks": zigzag_chunks,
             "cp_chunks_one_doc": cp_chunks_one_doc}


def make(name: str, seed: int | None = None, **kw) -> ThdBatch:
    fn = WORKLOADS[name]
    return fn(**kw) if seed is None else fn(seed=seed, **kw)


def random_pack(seed: int, *, batch: int = 4, max_len: int = 200, h_q: int = 4, h_kv: int = 2,
                d: int = 64, dtype: str = "bf16", max_gap: int = 9, stats_layout: int | None = None,
                masks=(0, 1, 2), with_qco: bool | None = None, allow_empty: bool = True,
                separate_kv_len: bool = True, nan_pads: bool = True,
                with_window: bool = False) -> ThdBatch:
    """Small random pack for fuzzing: ragged lengths, per-tensor gaps, mixed masks.

    Q/O/Stats share one set of offsets and K/V another, each with its own random
    gaps; query and key lengths differ per sequence when ``separate_kv_len``.
    """
    rng = np.random.default_rng(seed)
    lo = 0 if allow_empty else 1
    lq = rng.integers(lo, max_len, size=batch, endpoint=True)
    lk = rng.integers(lo, max_len, size=batch, endpoint=True) if separate_kv_len else lq.copy()
    gq = rng.integers(0, max_gap, size=batch, endpoint=True)
    gk = rng.integers(0, max_gap, size=batch, endpoint=True)
    lead_q, lead_k = int(rng.integers(0, 4)), int(rng.integers(0, 4))
    off_q = (_cumsum0(lq + gq) + lead_q).astype(np.int32)
    off_k = (_cumsum0(lk + gk) + lead_k).astype(np.int32)
    cap_q, cap_k = int(off_q[-1]) + int(rng.integers(0, 3)), int(off_k[-1]) + int(rng.integers(0, 3))
    q = _normal(rng, (cap_q, h_q, d), dtype)
    k = _normal(rng, (cap_k, h_kv, d), dtype)
    v = _normal(rng, (cap_k, h_kv, d), dtype)
    if nan_pads:
        _fill_rows(q, _pad_rows(cap_q, off_q[:-1], lq), float("nan"))
        pk = _pad_rows(cap_k, off_k[:-1], lk)
        _fill_rows(k, pk, float("nan"))
        _fill_rows(v, pk, float("nan"))
    mask = rng.choice(np.array(masks, dtype=np.int8), size=batch)
    if with_qco is None:
        with_qco = bool(rng.integers(0, 2))
    qco = None
    if with_qco:
        # any shift from "all rows dead" to "all keys visible"
        qco = np.array([int(rng.integers(-int(a) - 2, int(b_) + 2)) for a, b_ in zip(lq, lk)],
                       dtype=np.int32)
    if stats_layout is None:
        stats_layout = int(rng.integers(0, 2))
    window = None
    if with_window:
        # unbounded (-1), zero, and windows shorter and longer than the sequence
        window = np.array([int(rng.choice([-1, 0, int(rng.integers(1, max_len + 2)), 3 * max_len]))
                           for _ in range(batch)], dtype=np.int32)
    return ThdBatch(f"random_pack_{seed}", dtype, h_q, h_kv, d, _cumsum0(lq), _cumsum0(lk),
                    off_q, off_k, off_k.copy(), off_q.copy(), off_q.copy(), mask, qco,
                    stats_layout, q, k, v, cap_q, cap_q, window_left=window)


# ------------------------------------------------------------------- indexer inputs
@dataclass
class IndexerBatch:
    """Packed inputs of the sparse-attention indexer top-k: QI [cap_q, H, d],
    KI [cap_k, d], W [cap_q, H] float32 (rows addressed like QI's), and the
    output rows ``off_out`` of an int32 [cap_out, topk] index tensor."""
    name: str
    dtype: str
    heads: int
    d: int
    topk: int
    cu_seqlens_q: np.ndarray
    cu_seqlens_kv: np.ndarray
    off_q: np.ndarray
    off_k: np.ndarray
    off_out: np.ndarray
    mask_type: np.ndarray
    q_causal_offset: np.ndarray | None
    q: torch.Tensor
    k: torch.Tensor
    w: torch.Tensor
    cap_out: int

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens_q) - 1

    def lens_q(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)

    def lens_k(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_kv)


INDEXER_CP_SEED = 106


def indexer_cp(seed: int = INDEXER_CP_SEED, docs: int = 2, k_len: int = 65536, q_len: int = 4096, heads: int = 64,
               d: int = 128, topk: int = 2048, dtype: str = "bf16") -> IndexerBatch:
    """Context-parallel indexer chunks (the Megatron-LM PR #14 multi-document case):
    per document a packed key prefix of ``k_len`` tokens and a ``q_len``-row query
    chunk at causal offset k_len - q_len (bottom-right), N(0,1) indexer vectors,
    weights N(0,1)/sqrt(H)."""
    rng = np.random.default_rng(seed)
    lq = np.full(docs, q_len, dtype=np.int64)
    lk = np.full(docs, k_len, dtype=np.int64)
    off_q = _cumsum0(lq)[:-1].astype(np.int32)
    off_k = _cumsum0(lk)[:-1].astype(np.int32)
    q = _normal(rng, (int(lq.sum()), heads, d), dtype)
    k = _normal(rng, (int(lk.sum()), d), dtype)
    w = torch.from_numpy((rng.standard_normal((int(lq.sum()), heads)) / np.sqrt(heads)).astype(np.float32))
    return IndexerBatch("indexer_cp", dtype, heads, d, topk, _cumsum0(lq), _cumsum0(lk), off_q, off_k,
                        off_q.copy(), np.full(docs, MASK_BOTTOM_RIGHT, dtype=np.int8),
                        (lk - lq).astype(np.int32), q, k, w, int(lq.sum()))


def indexer_random_pack(seed: int, *, batch: int = 4, max_len: int = 300, heads: int = 4, d: int = 64,
                        topk: int = 16, dtype: str = "bf16", masks=(0, 1, 2), max_gap: int = 5,
                        zero_q_rows: int = 0) -> IndexerBatch:
    """Small random indexer pack: ragged lengths, gaps in QI, KI and the output,
    mixed masks and causal offsets; ``zero_q_rows`` rows get q = 0 (every score 0:
    the selection is decided by the tie order alone)."""
    rng = np.random.default_rng(seed)
    lq = rng.integers(0, max_len, size=batch, endpoint=True)
    lk = rng.integers(0, max_len, size=batch, endpoint=True)
    gq = rng.integers(0, max_gap, size=batch, endpoint=True)
    gk = rng.integers(0, max_gap, size=batch, endpoint=True)
    go = rng.integers(0, max_gap, size=batch, endpoint=True)
    off_q = (_cumsum0(lq + gq) + 1).astype(np.int32)[:-1]
    off_k = (_cumsum0(lk + gk) + 2).astype(np.int32)[:-1]
    off_o = (_cumsum0(lq + go) + 3).astype(np.int32)[:-1]
    cap_q = int(off_q[-1] + lq[-1] + 2) if batch else 1
    cap_k = int(off_k[-1] + lk[-1] + 2) if batch else 1
    cap_o = int(off_o[-1] + lq[-1] + 2) if batch else 1
    q = _normal(rng, (cap_q, heads, d), dtype)
    k = _normal(rng, (cap_k, d), dtype)
    w = torch.from_numpy(rng.standard_normal((cap_q, heads)).astype(np.float32))
    if zero_q_rows:
        rows = rng.choice(cap_q, size=min(zero_q_rows, cap_q), replace=False)
        q[torch.from_numpy(rows)] = 0
    mask = rng.choice(np.array(masks, dtype=np.int8), size=batch)
    qco = np.array([int(rng.integers(-2, int(b_) + 3)) for b_ in lk], dtype=np.int32)
    return IndexerBatch(f"indexer_random_{seed}", dtype, heads, d, topk, _cumsum0(lq), _cumsum0(lk),
                        off_q, off_k, off_o, mask, qco, q, k, w, cap_o)


def indexer_zigzag(seed: int = 107, doc_len: int = 4096, cp_size: int = 2, ranks=(0, 1), heads: int = 8,
                   d: int = 64, topk: int = 64, dtype: str = "bf16") -> IndexerBatch:
    """Zigzag context-parallel query chunks of one document (Megatron-LM PR #14,
    the packed-CP indexer paths): the document is cut into 2 * cp_size chunks of
    doc_len / (2 * cp_size) rows and rank r holds chunks r and 2 * cp_size - 1 - r.
    Every chunk becomes one THD segment whose queries see the key prefix that ends
    with the chunk, bottom-right aligned at q_causal_offset = the chunk's first
    global row. All segments read the SAME key rows (off_k = 0), so the segments'
    key ranges overlap."""
    rng = np.random.default_rng(seed)
    c = doc_len // (2 * cp_size)
    chunks = [ch for r in ranks for ch in (r, 2 * cp_size - 1 - r)]
    lq = np.full(len(chunks), c, dtype=np.int64)
    lk = np.array([(ch + 1) * c for ch in chunks], dtype=np.int64)
    off_q = _cumsum0(lq)[:-1].astype(np.int32)
    q = _normal(rng, (int(lq.sum()), heads, d), dtype)
    k = _normal(rng, (doc_len, d), dtype)
    w = torch.from_numpy((rng.standard_normal((int(lq.sum()), heads)) / np.sqrt(heads)).astype(np.float32))
    return IndexerBatch(f"indexer_zigzag_{seed}", dtype, heads, d, topk, _cumsum0(lq), _cumsum0(lk), off_q,
                        np.zeros(len(chunks), dtype=np.int32), off_q.copy(),
                        np.full(len(chunks), MASK_BOTTOM_RIGHT, dtype=np.int8),
                        np.array([ch * c for ch in chunks], dtype=np.int32), q, k, w, int(lq.sum()))
