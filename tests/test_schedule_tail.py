"""Host-side rule of the KV split's last wave (the CPU mirror of the setup kernel):
which pairs are cut into more than two parts, and that doing so shortens a greedy
longest-first schedule of the units over the CTAs."""
from __future__ import annotations

import heapq

import schedule_mirror as sm

SMS = 152


def _makespan(entries, h_q: int, per_unit: float = 3.0) -> float:
    """Greedy list schedule (each unit to the CTA that frees first, longest first):
    a unit of c tiles takes per_unit + c."""
    units = sorted((c for *_, c in entries for _ in range(h_q)), reverse=True)
    free = [0.0] * SMS
    for c in units:
        t = heapq.heappop(free)
        heapq.heappush(free, t + per_unit + c)
    return max(free)


def _parts(entries):
    out = {}
    for b, r, _, n, _ in entries:
        out[(b, r)] = n
    return out


def test_equal_pairs_last_wave_cut_into_eight():
    # the 128k-token shape: 32 pairs of ~496 tiles, 16 heads: halves give 1024 units
    # = 6 waves + 112 units; 112 units are 7 half entries, i.e. 4 pairs
    pairs = [(e // 16, (e % 16) * 256, 496) for e in range(32)]
    entries, n_split = sm.split_entries(pairs, 16, SMS, 40, True)
    parts = _parts(entries)
    assert n_split == 32
    eight = sorted(k for k, n in parts.items() if n == 8)
    # equal costs: the pairs with the highest indices in the pair list
    assert eight == sorted((e // 16, (e % 16) * 256) for e in range(28, 32))
    assert sum(1 for n in parts.values() if n == 2) == 28
    assert len(entries) == 28 * 2 + 4 * 8
    halves_only = [x for b, r, c in pairs for x in ((b, r, 0, 2, c // 2), (b, r, 1, 2, c - c // 2))]
    assert _makespan(entries, 16) < 0.98 * _makespan(halves_only, 16)


def test_cheapest_pairs_taken_and_part_costs_sum():
    costs = [300 + 7 * e for e in range(32)]
    pairs = [(e, 0, c) for e, c in enumerate(costs)]
    entries, _ = sm.split_entries(pairs, 16, SMS, 40, True)
    parts = _parts(entries)
    assert sorted(b for (b, _), n in parts.items() if n == 8) == [0, 1, 2, 3]
    for e, c in enumerate(costs):
        got = sorted(x[2] for x in entries if x[0] == e)
        assert got == list(range(parts[(e, 0)]))
        assert sum(x[4] for x in entries if x[0] == e) == c


def test_ties_prefer_higher_index():
    # two cheapest costs tie across 6 pairs; 4 are needed: the 2 cheapest plus the
    # 2 highest-indexed of the next cost
    costs = [500] * 26 + [200, 200] + [300] * 4
    pairs = [(e, 0, c) for e, c in enumerate(costs)]
    entries, _ = sm.split_entries(pairs, 16, SMS, 40, True)
    eight = sorted(b for (b, _), n in _parts(entries).items() if n == 8)
    assert eight == [26, 27, 30, 31]


def test_no_tail_without_a_full_wave_or_below_min_cost():
    pairs = [(e, 0, 400) for e in range(4)]                   # 8 half entries x 16 = 128 units < 152
    entries, _ = sm.split_entries(pairs, 16, SMS, 40, True)
    assert set(_parts(entries).values()) == {2}
    pairs = [(e, 0, 60) for e in range(32)]                   # parts would fall below 8 tiles
    entries, _ = sm.split_entries(pairs, 16, SMS, 40, True)
    assert set(_parts(entries).values()) == {2}
    pairs = [(e, 0, 496) for e in range(19)]                   # halves: 608 units = 4 full waves
    entries, _ = sm.split_entries(pairs, 16, SMS, 40, True)
    assert set(_parts(entries).values()) == {2}


def test_tail_count_follows_last_wave_one_head():
    # one head: a unit per half entry, so the last wave's rest units give rest / 2
    # pairs (within the workspace's max_tail_pairs(1) = 80 pairs of extra slots)
    pairs = [(e, 0, 100) for e in range(200)]                 # 400 units: 2 waves + 96
    entries, _ = sm.split_entries(pairs, 1, SMS, 640, True)
    n8 = sum(1 for n in _parts(entries).values() if n == 8)
    assert n8 == 48
    pairs = [(e, 0, 100) for e in range(300)]                 # 600 units: 3 waves + 144 -> 72 pairs
    entries, _ = sm.split_entries(pairs, 1, SMS, 640, True)
    assert sum(1 for n in _parts(entries).values() if n == 8) == 72


def test_entries_and_slots_fit_the_plan_capacity():
    """The pair list holds max_pairs + max_split + 6 max_tail entries and the partial
    buffers 2 max_split + 6 max_tail slots (max_split = min(max_pairs, ceil(640 / h)),
    max_tail = min(max_split, ceil((ceil(160 / h) + 1) / 2))): no pair list the rule can
    see exceeds either, whatever the costs, heads and CTA count."""
    import numpy as np
    rng = np.random.default_rng(5)
    for _ in range(3000):
        h = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64]))
        max_pairs = int(rng.integers(1, 400))
        n = int(rng.integers(1, max_pairs + 1))
        hi = int(rng.choice([20, 70, 200, 600, 1500]))
        pairs = [(e, 0, int(c)) for e, c in enumerate(rng.integers(0, hi, size=n))]
        num_ctas = min(int(rng.choice([148, 152, 160])), 2 * max_pairs * h)
        max_split = min(max_pairs, -(-4 * 160 // h))
        max_tail = min(max_split, (-(-160 // h) + 1) // 2)
        entries, n_split = sm.split_entries(pairs, h, num_ctas, max_split, True)
        assert len(entries) <= max_pairs + max_split + 6 * max_tail
        slots = sum(1 for x in entries if x[3] > 1)
        assert slots <= 2 * max_split + 6 * max_tail
        assert sum(1 for x in entries if x[3] == 8) <= 8 * max_tail
