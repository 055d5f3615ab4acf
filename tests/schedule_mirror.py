"""CPU mirror of the setup kernel's outputs (metadata, pair list, header words).

The setup kernel's contract, restated independently: per sequence
``(len_q, len_k, off_q, off_k, off_v, off_o, off_s, shift, lo_shift, 0, 0, 0)``; invalid
sequences (negative length, offset outside capacity, unknown mask) get
``len_q = 0`` and a status bit; every valid sequence contributes
``ceil(len_q / rows_per_unit)`` pairs ``(b, row0)``, ordered by descending cost
(KV tiles to visit, clamped to the bucket count) -- the order inside one cost
bucket is not fixed.
"""
from __future__ import annotations

import numpy as np

COST_BINS = 1024
COST_GROUPS = 11
NO_LOWER_BOUND = -(1 << 30)


def cost_group(c: int) -> int:
    """0 for costs 512..1023, 1 for 256..511, ..., 9 for 1, 10 for 0."""
    return COST_GROUPS - 1 if c == 0 else 9 - (int(c).bit_length() - 1)


def group_starts(pairs) -> list[int]:
    """First pair index of each cost group in the longest-first list, plus the count."""
    counts = [0] * COST_GROUPS
    for _, _, c in pairs:
        counts[cost_group(c)] += 1
    out, acc = [], 0
    for n in counts:
        out.append(acc)
        acc += n
    return out + [acc]


def unit_order(starts, h_q: int, h_kv: int):
    """(pair index, query head) of every work id: inside a cost group kv head, then
    pair, then query head of the kv group."""
    grp = h_q // h_kv
    out = []
    for g in range(COST_GROUPS):
        a, b = starts[g], starts[g + 1]
        for kvh in range(h_kv):
            for pr in range(a, b):
                for hh in range(grp):
                    out.append((pr, kvh * grp + hh))
    return out


BAD_LENGTH, BAD_OFFSET, BAD_MASK, TILE_OVERFLOW = 1, 2, 4, 8


SPLIT_WAVES, MIN_SPLIT_COST = 4, 16
TAIL_PARTS, MIN_TAIL_COST, MAX_SMS_FOR_SIZING = 8, 64, 160


def part_cost(cost: int, i: int, n: int) -> int:
    """Tiles of part i of a pair of `cost` tiles cut into n parts."""
    return (i + 1) * cost // n - i * cost // n


def split_entries(pairs, h_q: int, num_ctas: int, max_split: int, allow_split: bool):
    """Scheduled entries after the KV-split decision: list of (b, row0, part, parts,
    cost) and the number of split pairs. Pairs visiting at least MIN_SPLIT_COST KV
    tiles are halved when the launch has fewer than SPLIT_WAVES waves of units. When
    the halves leave a partial last wave after at least one full one, the cheapest
    split pairs that fill it (ascending cost, then descending index in the pair list)
    are cut into TAIL_PARTS parts, provided the threshold cost is at least
    MIN_TAIL_COST and below the clamped top bucket; pairs below MIN_TAIL_COST keep two."""
    splittable = [p for p in pairs if p[2] >= MIN_SPLIT_COST]
    on = (allow_split and len(pairs) > 0 and len(pairs) * h_q < SPLIT_WAVES * num_ctas
          and 0 < len(splittable) <= max_split)
    tail = set()
    if on:
        units = (len(pairs) + len(splittable)) * h_q
        rest = units % num_ctas
        if units >= num_ctas and rest > 0:
            max_tail = min(max_split, (-(-MAX_SMS_FOR_SIZING // h_q) + 1) // 2)
            need = min((-(-rest // h_q) + 1) // 2, max_tail)
            cand = sorted((c, -e) for e, (_, _, c) in enumerate(pairs) if c >= MIN_SPLIT_COST)
            if 0 < need <= len(cand) and MIN_TAIL_COST <= cand[need - 1][0] < COST_BINS - 1:
                tail = {-ne for c, ne in cand[:need] if c >= MIN_TAIL_COST}
    out = []
    for e, (b, r, c) in enumerate(pairs):
        n = 1 if not (on and c >= MIN_SPLIT_COST) else (TAIL_PARTS if e in tail else 2)
        if n == 1:
            out.append((b, r, 0, 1, c))
        else:
            out.extend((b, r, i, n, min(part_cost(c, i, n), COST_BINS - 1)) for i in range(n))
    return out, (len(splittable) if on else 0)


def mirror(batch, rows_per_unit: int, keys_per_tile: int, max_pairs: int, caps=None):
    """Expected (meta [B, 12] int32, pairs list of (b, row0, cost), status, num_pairs).
    Costs are the KV-tile counts (first visible tile of the pair's first row through
    the last of its last row) clamped to the bucket range."""
    lq = batch.lens_q()
    lk = batch.lens_k()
    if caps is None:
        caps = (batch.q.shape[0], batch.k.shape[0], batch.v.shape[0], batch.cap_o, batch.cap_s)
    cap_q, cap_k, cap_v, cap_o, cap_s = caps
    meta = np.zeros((batch.batch, 12), dtype=np.int64)
    status = 0
    pairs = []
    for b in range(batch.batch):
        offs = [int(x[b]) for x in (batch.off_q, batch.off_k, batch.off_v, batch.off_o, batch.off_s)]
        mt = int(batch.mask_type[b])
        bad = 0
        if lq[b] < 0 or lk[b] < 0:
            bad |= BAD_LENGTH
        if mt not in (0, 1, 2):
            bad |= BAD_MASK
        if not bad:
            lens = (lq[b], lk[b], lk[b], lq[b], lq[b])
            for off, n, cap in zip(offs, lens, (cap_q, cap_k, cap_v, cap_o, cap_s)):
                if off < 0 or off + n > cap:
                    bad |= BAD_OFFSET
        if mt == 0:
            shift = int(lk[b])
        elif mt == 1:
            shift = 0
        else:
            shift = int(lk[b] - lq[b]) if batch.q_causal_offset is None else int(batch.q_causal_offset[b])
        lo = NO_LOWER_BOUND
        win = None if batch.window_left is None else int(batch.window_left[b])
        if win is not None and win >= 0 and mt in (1, 2):
            lo = max(NO_LOWER_BOUND, min(1 << 30, shift - win))
        shift = max(-(1 << 30), min(1 << 30, shift))
        meta[b] = [0 if bad else lq[b], lk[b], *offs, shift, lo, 0, 0, 0]
        status |= bad
        if bad:
            continue
        for t in range((int(lq[b]) + rows_per_unit - 1) // rows_per_unit):
            row0 = t * rows_per_unit
            r_end = min(int(lq[b]), row0 + rows_per_unit)
            kmax = min(int(lk[b]), r_end + shift)
            first = max(0, row0 + lo) // keys_per_tile
            cost = 0 if kmax <= 0 else max(0, (kmax + keys_per_tile - 1) // keys_per_tile - first)
            pairs.append((b, row0, min(cost, COST_BINS - 1)))
    if len(pairs) > max_pairs:
        status |= TILE_OVERFLOW
        pairs = []
    return meta.astype(np.int32), pairs, status, len(pairs)
