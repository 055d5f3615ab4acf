// Setup kernel: turns the caller's device-resident lengths and per-tensor ragged
// offsets into per-sequence metadata and a longest-first list of query tiles,
// with no device-to-host read (cuDNN-frontend issue "THD lowering never reads the
// bound ragged offsets", section "Proposal: consume the bound offsets on device";
// TransformerEngine PR #3274 review: avoid GPU-CPU syncs so the call stays graph
// capturable).
//
// One block of 1024 threads:
//   1. per sequence: lengths from cu_seqlens, offsets read as bound, validation,
//      causal shift; block scan of the per-sequence tile counts;
//   2. histogram of tile costs (KV tiles to visit) in kCostBins buckets;
//   3. descending exclusive scan of the histogram (longest tiles first);
//   4. scatter of every (sequence, first row) pair to its bucket's next slot.
// When a launch has fewer than kSplitWaves waves of units and splitting is
// allowed, long pairs are scheduled as two halves of their KV range (two entries,
// a partial-result slot each, one record for the combine kernel), which evens out
// the persistent grid; if the halves still leave a partial last wave, the cheapest
// split pairs whose units would make it up are cut into kTailParts parts instead,
// so short units fill the end of the launch. Entries and partial slots are checked
// against the plan's capacities before anything is written.
// It also zeroes the persistent scheduler's tile counter (header word 0) and
// writes the status word, pair count and tile count. Invalid sequences get no
// tiles and set a status bit; their rows are never touched.
// On the backward's key axis (units over keys for dK/dV), consecutive sequences
// that read the same K and V rows -- the zigzag query chunks of one document under
// context parallelism (Megatron-LM PR #14, the packed-CP paths) -- form one key
// group: its units cover the group's keys and sum the gradient of every member,
// and key rows shared in any other way are reported (THD_DEV_KEY_OVERLAP) instead
// of racing.
#include "internal.h"

namespace thd {

namespace {

__device__ __forceinline__ int32_t block_inclusive_scan(int32_t x, int32_t* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int32_t r = x + (warp > 0 ? warp_sums[warp - 1] : 0);
  __syncthreads();  // warp_sums may be reused by the caller's next scan
  return r;
}

// number of KV tiles the pair starting at row0 must visit: from the tile of the
// first row's lowest visible key to the tile of the last row's highest
__device__ __forceinline__ int32_t query_pair_cost(const SeqMeta& m, int32_t row0, int32_t rows_per_unit,
                                                   int32_t keys_per_tile) {
  const int64_t r_end = min64((int64_t)m.len_q, (int64_t)row0 + rows_per_unit);
  const int64_t kmax = min64((int64_t)m.len_k, r_end + (int64_t)m.shift);
  if (kmax <= 0) return 0;
  const int64_t kmin = max64(0, (int64_t)row0 + (int64_t)m.lo_shift);
  const int64_t first = kmin / keys_per_tile, end = (kmax + keys_per_tile - 1) / keys_per_tile;
  return (int32_t)max64(0, end - first);
}

// key axis (backward dK/dV units): number of query tiles of `rows_per_tile` rows
// that see any key of [k0, k0 + keys_per_unit): key j is seen by rows
// j - shift <= i <= j - lo_shift
__device__ __forceinline__ int32_t key_pair_cost(const SeqMeta& m, int32_t k0, int32_t keys_per_unit,
                                                 int32_t rows_per_tile) {
  const int64_t k_end = min64((int64_t)m.len_k, (int64_t)k0 + keys_per_unit);
  if (k_end <= k0) return 0;
  const int64_t i_lo = max64(0, (int64_t)k0 - (int64_t)m.shift);
  const int64_t i_hi = min64((int64_t)m.len_q, (k_end - 1) - (int64_t)m.lo_shift + 1);
  if (i_hi <= i_lo) return 0;
  return (int32_t)((i_hi + rows_per_tile - 1) / rows_per_tile - i_lo / rows_per_tile);
}

// cost of the unit whose pair starts at row0 of sequence b; with key groups the
// query tiles of every valid member of b's group
__device__ __forceinline__ int32_t pair_cost(const SetupParams& p, int32_t b, int32_t row0) {
  const SeqMeta m = p.meta[b];
  if (!p.key_axis) return query_pair_cost(m, row0, p.rows_per_unit, p.keys_per_tile);
  if (!p.group_keys) return key_pair_cost(m, row0, p.rows_per_unit, p.keys_per_tile);
  int32_t c = 0;
  for (int32_t e = b; e < b + m.group_n; ++e) {
    const SeqMeta me = p.meta[e];
    if (me.bad == 0) c += key_pair_cost(me, row0, p.rows_per_unit, p.keys_per_tile);
  }
  return c;
}

__device__ __forceinline__ int64_t block_inclusive_max(int64_t x, int64_t* warp_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max64(x, y);
  }
  if (lane == 31) warp_max[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t s = warp_max[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s = max64(s, y);
    }
    warp_max[lane] = s;
  }
  __syncthreads();
  const int64_t r = warp > 0 ? max64(x, warp_max[warp - 1]) : x;
  __syncthreads();
  return r;
}

// sequence e reads the same K and V rows as sequence e - 1
__device__ __forceinline__ bool same_keys(const SetupParams& p, int32_t e) {
  return e > 0 && p.off_k[e] == p.off_k[e - 1] && p.off_v[e] == p.off_v[e - 1];
}

// tiles of part i of a pair of `cost` tiles cut into n parts ([i c / n, (i + 1) c / n))
__device__ __forceinline__ int32_t part_cost(int32_t cost, int32_t i, int32_t n) {
  return (int32_t)(((int64_t)(i + 1) * cost) / n - ((int64_t)i * cost) / n);
}

// group of a (clamped) cost: 0 for 512..1023, 1 for 256..511, ..., 9 for 1, 10 for 0
__device__ __forceinline__ int cost_group(int32_t c) { return c == 0 ? kCostGroups - 1 : 9 - (31 - __clz(c)); }

__device__ __forceinline__ int32_t find_seq(const int32_t* pair_base, int32_t batch, int32_t e) {
  // last b with pair_base[b] <= e (pair_base is non-decreasing, pair_base[0] == 0)
  int32_t lo = 0, hi = batch;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (pair_base[mid] <= e) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kSetupThreads) setup_kernel(SetupParams p) {
  __shared__ uint32_t hist[kCostBins];
  __shared__ uint32_t group_count[kCostGroups];
  __shared__ uint32_t n_splittable, n_split_done, n_slots, n_slots_need;
  __shared__ bool split_on, sched_ok;
  __shared__ int32_t tail_need, tail_cost, tail_ties, tail_tie_count, tail_e, tie_seen;
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  __shared__ uint32_t status_s;
  const int tid = threadIdx.x;
  for (int i = tid; i < kCostBins; i += blockDim.x) hist[i] = 0;
  if (tid < kCostGroups) group_count[tid] = 0;
  if (tid == 0) { carry = 0; status_s = 0; n_splittable = 0; }
  __syncthreads();

  // 1. per-sequence metadata and tile counts
  for (int32_t base = 0; base < p.batch; base += blockDim.x) {
    const int32_t b = base + tid;
    int32_t n = 0;
    if (b < p.batch) {
      const int32_t lq = p.cu_q[b + 1] - p.cu_q[b];
      const int32_t lk = p.cu_k[b + 1] - p.cu_k[b];
      SeqMeta m;
      m.len_q = lq; m.len_k = lk;
      uint32_t bad = 0;
      const int32_t* offs[5] = {p.off_q, p.off_k, p.off_v, p.off_o, p.off_s};
      int32_t rows[5];
#pragma unroll
      for (int x = 0; x < 5; ++x) {
        int64_t v = (int64_t)offs[x][b];
        if (p.element_offsets) {
          // element offset (x multiplier) -> row: must be a whole number of rows
          v *= p.offset_multiplier;
          if (v < 0 || v % p.tok_stride[x] != 0 || v / p.tok_stride[x] > 0x7fffffffll) bad |= THD_DEV_BAD_OFFSET;
          v = v / p.tok_stride[x];
        }
        rows[x] = (int32_t)v;
      }
      m.off_q = rows[0]; m.off_k = rows[1]; m.off_v = rows[2]; m.off_o = rows[3]; m.off_s = rows[4];
      const int mt = (int)p.mask[b];
      if (lq < 0 || lk < 0 || (p.max_len_k > 0 && lk > p.max_len_k)) bad |= THD_DEV_BAD_LENGTH;
      if (mt < 0 || mt > 2) bad |= THD_DEV_BAD_MASK;
      if (!bad) {
        auto in_cap = [](int32_t off, int32_t len, int64_t cap) {
          return off >= 0 && (int64_t)off + (int64_t)len <= cap;
        };
        if (!in_cap(m.off_q, lq, p.cap_q) || !in_cap(m.off_k, lk, p.cap_k) ||
            !in_cap(m.off_v, lk, p.cap_v) || !in_cap(m.off_o, lq, p.cap_o) ||
            !in_cap(m.off_s, lq, p.cap_s))
          bad |= THD_DEV_BAD_OFFSET;
      }
      int64_t shift;
      if (mt == THD_MASK_NONE) shift = lk;
      else if (mt == THD_MASK_CAUSAL_TOP_LEFT) shift = 0;
      else shift = p.qco ? (int64_t)p.qco[b] : (int64_t)lk - (int64_t)lq;
      // left window of the causal masks: row i also needs j >= i + shift - w
      int64_t lo = kNoLowerBound;
      if (p.window && mt != THD_MASK_NONE && p.window[b] >= 0) lo = shift - (int64_t)p.window[b];
      // beyond +-2^30 a shift no longer changes which keys are visible
      shift = max64(-(1ll << 30), min64(1ll << 30, shift));
      lo = max64(kNoLowerBound, min64(1ll << 30, lo));
      m.shift = (int32_t)shift;
      m.lo_shift = (int32_t)lo;
      m.group_n = p.group_keys ? 1 : 0;
      m.group_len_k = 0;
      m.bad = p.group_keys ? (int32_t)bad : 0;
      if (bad) {
        atomicOr(&status_s, bad);
        m.len_q = 0;  // no tiles, rows untouched
      } else {
        n = ((p.key_axis ? lk : lq) + p.rows_per_unit - 1) / p.rows_per_unit;
      }
      p.meta[b] = m;
    }
    const int32_t incl = block_inclusive_scan(n, warp_sums);
    if (b < p.batch) p.pair_base[b] = carry + incl - n;
    __syncthreads();
    if (tid == blockDim.x - 1) carry += incl;
    __syncthreads();
  }
  if (p.group_keys) {
    // 1b. key groups: a run of consecutive sequences with equal K and V offsets is
    // one group, scheduled from its first member over the longest valid member's
    // keys; the other members get no pairs of their own
    __syncthreads();   // every sequence's metadata is written
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int32_t base = 0; base < p.batch; base += blockDim.x) {
      const int32_t b = base + tid;
      int32_t n = 0;
      if (b < p.batch) {
        SeqMeta* mb = p.meta + b;
        if (same_keys(p, b)) {
          mb->group_n = 0;
        } else {
          int32_t cnt = 1, glen = mb->bad == 0 ? mb->len_k : 0;
          for (int32_t e = b + 1; e < p.batch && same_keys(p, e); ++e, ++cnt)
            if (p.meta[e].bad == 0) glen = max(glen, p.meta[e].len_k);
          mb->group_n = cnt;
          mb->group_len_k = glen;
          n = (glen + p.rows_per_unit - 1) / p.rows_per_unit;
        }
      }
      const int32_t incl = block_inclusive_scan(n, warp_sums);
      if (b < p.batch) p.pair_base[b] = carry + incl - n;
      __syncthreads();
      if (tid == blockDim.x - 1) carry += incl;
      __syncthreads();
    }
    // 1c. the K rows (and the V rows) of different groups must be disjoint: their
    // dK/dV units would race otherwise. With group starts non-decreasing in batch
    // order (packed layouts), a group overlaps an earlier one exactly when it starts
    // before the largest end seen so far; otherwise every pair of groups is checked.
    __shared__ int64_t warp_max[32];
    __shared__ int64_t run_start[2], run_end[2];
    __shared__ int unsorted;
    if (tid == 0) { run_start[0] = run_start[1] = run_end[0] = run_end[1] = INT64_MIN; unsorted = 0; }
    __syncthreads();
    uint32_t overlap = 0;
    for (int32_t base = 0; base < p.batch; base += blockDim.x) {
      const int32_t b = base + tid;
      bool lead = false;
      SeqMeta m;
      if (b < p.batch) {
        m = p.meta[b];
        lead = m.group_n > 0 && m.group_len_k > 0;
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int64_t st = lead ? (int64_t)(x == 0 ? m.off_k : m.off_v) : INT64_MIN;
        const int64_t en = lead ? st + m.group_len_k : INT64_MIN;
        const int64_t max_st = block_inclusive_max(st, warp_max);
        const int64_t max_en_incl = block_inclusive_max(en, warp_max);
        // exclusive maxima: shift by one thread through shared memory
        __shared__ int64_t ex_st[kSetupThreads], ex_en[kSetupThreads];
        ex_st[tid] = max_st;
        ex_en[tid] = max_en_incl;
        __syncthreads();
        const int64_t prev_st = max64(run_start[x], tid > 0 ? ex_st[tid - 1] : INT64_MIN);
        const int64_t prev_en = max64(run_end[x], tid > 0 ? ex_en[tid - 1] : INT64_MIN);
        if (lead) {
          if (st < prev_st) unsorted = 1;
          else if (st < prev_en) overlap = 1;
        }
        __syncthreads();
        if (tid == blockDim.x - 1) {
          run_start[x] = max64(run_start[x], max_st);
          run_end[x] = max64(run_end[x], max_en_incl);
        }
        __syncthreads();
      }
    }
    if (unsorted) {
      for (int32_t b = tid; b < p.batch; b += blockDim.x) {
        const SeqMeta m = p.meta[b];
        if (m.group_n == 0 || m.group_len_k == 0) continue;
        for (int32_t e = b + 1; e < p.batch && !overlap; ++e) {
          const SeqMeta o = p.meta[e];
          if (o.group_n == 0 || o.group_len_k == 0) continue;
          const bool k_ov = (int64_t)m.off_k < (int64_t)o.off_k + o.group_len_k &&
                            (int64_t)o.off_k < (int64_t)m.off_k + m.group_len_k;
          const bool v_ov = (int64_t)m.off_v < (int64_t)o.off_v + o.group_len_k &&
                            (int64_t)o.off_v < (int64_t)m.off_v + m.group_len_k;
          if (k_ov || v_ov) overlap = 1;
        }
      }
    }
    if (overlap) atomicOr(&status_s, (uint32_t)THD_DEV_KEY_OVERLAP);
    __syncthreads();
    if (status_s & THD_DEV_KEY_OVERLAP) carry = 0;   // no dK/dV units at all
    __syncthreads();
  }
  int32_t total = carry;
  if (tid == 0) p.pair_base[p.batch] = total;
  if (total > p.max_pairs) {
    if (tid == 0) atomicOr(&status_s, (uint32_t)THD_DEV_TILE_OVERFLOW);
    total = 0;
  }
  __syncthreads();

  // 2a. KV split decision: with fewer than kSplitWaves waves of units, pairs that
  // visit at least kMinSplitCost KV tiles are processed as two halves
  for (int32_t e = tid; e < total; e += blockDim.x) {
    const int32_t b = find_seq(p.pair_base, p.batch, e);
    const int32_t row0 = (e - p.pair_base[b]) * p.rows_per_unit;
    if (pair_cost(p, b, row0) >= kMinSplitCost) atomicAdd(&n_splittable, 1u);
  }
  __syncthreads();
  if (tid == 0) {
    split_on = p.allow_split && total > 0 &&
               (int64_t)total * p.unit_heads < (int64_t)kSplitWaves * p.num_ctas && n_splittable > 0 &&
               (int32_t)n_splittable <= p.max_split;
    n_split_done = 0;
    n_slots = 0;
    n_slots_need = 0;
    tail_cost = -1;
    tail_ties = tail_tie_count = 0;
    tail_e = 0;
    tie_seen = 0;
    // units of a last, partial wave after halving: the `need` cheapest split pairs
    // (costs ascending, then the highest pair index first) are cut into kTailParts
    tail_need = 0;
    if (split_on) {
      const int64_t units = ((int64_t)total + n_splittable) * p.unit_heads;
      const int64_t rest = units % p.num_ctas;
      if (units >= p.num_ctas && rest > 0) {
        const int64_t entries = (rest + p.unit_heads - 1) / p.unit_heads;
        tail_need = (int32_t)min64((entries + 1) / 2, (int64_t)p.max_tail);
      }
    }
  }
  __syncthreads();

  // 2a'. tail pairs: cost histogram of the split pairs (one bucket per thread), an
  // inclusive scan finds the cost c_t at which `need` pairs are reached; among pairs
  // of cost c_t the ones with the highest index are taken (threshold index tail_e)
  if (tail_need > 0) {
    for (int32_t e = tid; e < total; e += blockDim.x) {
      const int32_t b = find_seq(p.pair_base, p.batch, e);
      const int32_t row0 = (e - p.pair_base[b]) * p.rows_per_unit;
      const int32_t c = pair_cost(p, b, row0);
      if (c >= kMinSplitCost) atomicAdd(&hist[min(c, kCostBins - 1)], 1u);
    }
    __syncthreads();
    const int32_t cnt = (int32_t)hist[tid];
    const int32_t incl = block_inclusive_scan(cnt, warp_sums);
    if (incl >= tail_need && incl - cnt < tail_need) {
      // the cheapest tail pairs must be long enough for kTailParts parts; the
      // clamped top bucket cannot order its pairs, so it takes no tail split
      if (tid >= kMinTailCost && tid < kCostBins - 1) {
        tail_cost = tid;
        tail_ties = tail_need - (incl - cnt);   // pairs of cost c_t to take
        tail_tie_count = cnt;
      }
    }
    __syncthreads();
    hist[tid] = 0;
    if (tail_cost >= 0 && tail_ties < tail_tie_count) {
      // rank the pairs of cost c_t by index, from the end: the tail_ties highest are taken
      for (int32_t base = 0; base < total; base += blockDim.x) {
        const int32_t e = base + tid;
        int32_t tie = 0;
        if (e < total) {
          const int32_t b = find_seq(p.pair_base, p.batch, e);
          const int32_t row0 = (e - p.pair_base[b]) * p.rows_per_unit;
          tie = pair_cost(p, b, row0) == tail_cost ? 1 : 0;
        }
        const int32_t incl_t = block_inclusive_scan(tie, warp_sums);
        const int32_t rank = tie_seen + incl_t - 1;      // among the ties, from the front
        if (tie && tail_tie_count - 1 - rank == tail_ties - 1) tail_e = e;
        __syncthreads();
        if (tid == blockDim.x - 1) tie_seen += incl_t;
        __syncthreads();
      }
    }
    __syncthreads();
  }
  // parts of a pair of cost c at index e (pairs below kMinTailCost keep two)
  auto parts_of = [&](int32_t c, int32_t e) -> int32_t {
    if (!split_on || c < kMinSplitCost) return 1;
    if (tail_cost >= 0 && c >= kMinTailCost && (c < tail_cost || (c == tail_cost && e >= tail_e)))
      return kTailParts;
    return 2;
  };

  // 2b. cost histogram over the scheduled entries (a pair in n parts gives n)
  for (int32_t e = tid; e < total; e += blockDim.x) {
    const int32_t b = find_seq(p.pair_base, p.batch, e);
    const int32_t row0 = (e - p.pair_base[b]) * p.rows_per_unit;
    const int32_t cost = pair_cost(p, b, row0);
    const int32_t n = parts_of(cost, e);
    if (n > 1) atomicAdd(&n_slots_need, (uint32_t)n);
    for (int32_t i = 0; i < n; ++i) {
      const int32_t c = min(part_cost(cost, i, n), kCostBins - 1);
      atomicAdd(&hist[c], 1u);
      atomicAdd(&group_count[cost_group(c)], 1u);
    }
  }
  __syncthreads();
  // the pair list and the partial slots are sized at plan time for every entry; a
  // schedule that does not fit is a TILE_OVERFLOW and gets no work at all
  if (tid == 0) {
    uint32_t entries = 0;
    for (int g = 0; g < kCostGroups; ++g) entries += group_count[g];
    sched_ok = entries <= (uint32_t)p.pair_cap && n_slots_need <= (uint32_t)max(p.slot_cap, 0);
    if (!sched_ok) {
      atomicOr(&status_s, (uint32_t)THD_DEV_TILE_OVERFLOW);
      for (int g = 0; g < kCostGroups; ++g) group_count[g] = 0;
    }
  }
  __syncthreads();

  // 3. exclusive scan from the most expensive bucket down
  for (int i = tid; i < kCostBins; i += blockDim.x) {
    // kCostBins == blockDim.x: one bucket per thread
    const int32_t cnt = (int32_t)hist[kCostBins - 1 - i];
    const int32_t incl = block_inclusive_scan(cnt, warp_sums);
    hist[kCostBins - 1 - i] = (uint32_t)(incl - cnt);
  }
  __syncthreads();

  // 4. scatter
  for (int32_t e = tid; sched_ok && e < total; e += blockDim.x) {
    const int32_t b = find_seq(p.pair_base, p.batch, e);
    const int32_t row0 = (e - p.pair_base[b]) * p.rows_per_unit;
    const int32_t cost = pair_cost(p, b, row0);
    const int32_t n = parts_of(cost, e);
    if (n > 1) {
      const int32_t part = (int32_t)atomicAdd(&n_split_done, 1u);
      const int32_t slot0 = (int32_t)atomicAdd(&n_slots, (uint32_t)n);
      SplitRec sr;
      sr.b = b; sr.row0 = row0; sr.slot0 = slot0; sr.parts = n;
      p.splits[part] = sr;
      for (int32_t i = 0; i < n; ++i) {
        const int32_t c = min(part_cost(cost, i, n), kCostBins - 1);
        const uint32_t slot = atomicAdd(&hist[c], 1u);
        PairRec r;
        r.b = b; r.row0 = row0; r.split = (i << 8) | n; r.part = slot0 + i;
        p.pairs[slot] = r;
      }
    } else {
      const int32_t c = min(cost, kCostBins - 1);
      const uint32_t slot = atomicAdd(&hist[c], 1u);
      PairRec r;
      r.b = b; r.row0 = row0; r.split = 1; r.part = -1;
      p.pairs[slot] = r;
    }
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t acc = 0;
    for (int g = 0; g < kCostGroups; ++g) {
      p.header[kHdrGroupStart + g] = acc;
      acc += group_count[g];
    }
    p.header[kHdrGroupStart + kCostGroups] = acc;   // entries after splitting
    p.header[kHdrCounter] = 0u;
    p.header[kHdrStatus] = status_s;
    p.header[kHdrNumPairs] = acc;
    p.header[kHdrNumTiles] = acc * (uint32_t)p.unit_heads;
    p.header[kHdrNumSplit] = split_on && sched_ok ? n_splittable : 0u;
  }
}

}  // namespace

cudaError_t launch_setup(const SetupParams& p, cudaStream_t stream) {
  static_assert(kCostBins == kSetupThreads, "one histogram bucket per thread in the scan");
  setup_kernel<<<1, kSetupThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace thd
