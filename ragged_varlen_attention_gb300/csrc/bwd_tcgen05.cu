// Tensor-core backward kernels for sm_103a: dQ per query tile and dK/dV per key
// tile, each a persistent warp-specialised kernel like the forward one (TMA
// producer thread, one MMA-issuing thread, two softmax warpgroups, TMEM
// accumulators), over the same ragged metadata and longest-first schedules.
//
// Gradients (ragged SDPA backward, NVIDIA/cudnn-frontend PR #462, "What" and
// "Root cause"), base 2: P = 2^(s * scale * log2 e - LSE2) on visible keys,
// dS = P (dP - D) with dP = dO V^T and D = <dO, O> per query row (both LSE2 and D
// come from the preprocess kernel), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
//
// dQ kernel (unit = 128 query rows x one query head; loop over KV tiles j):
//   S = Q K_j^T and dP = dO V_j^T (A and B K-major in shared memory) into TMEM;
//   the softmax warps read S (then release it, so S(j+1) can be issued at once),
//   form P in registers, read dP, and write dS (16-bit) back into dP's columns;
//   dQ += dS K_j (A = dS from TMEM, B = K_j read MN-major).
//   Issue order S(j), dP(j) | S(j+1) | dQ(j), dP(j+1) | ...: S(j+1) runs while the
//   softmax forms dS(j), and dQ(j) + dP(j+1) run while it forms P(j+1).
// dK/dV kernel (unit = 128 keys x one kv head; loop over the query heads of the
// kv group and the query tiles i that see the keys):
//   S^T = K Q_i^T and dP^T = V dO_i^T into TMEM (lanes = keys); the softmax warps
//   write P^T (16-bit) over S^T and dS^T over dP^T; dV += P^T dO_i and
//   dK += dS^T Q_i (A from TMEM, B = dO_i / Q_i read MN-major). Per-column LSE2
//   and D arrive with Q_i as one 1 KB bulk copy. dK and dV are complete sums over
//   the group's heads: no atomics.
//   Issue order S(i), dP(i) | dV(i), S(i+1) | dK(i), dP(i+1) | ...
//
// TMEM (512 columns): S [0,128), dP [128,256), accumulators from 256 (dQ: D
// columns; dV then dK: D each). The two softmax warpgroups split the 128 columns
// of S and dP (64 each); each writes its 16-bit P or dS into the first 32 columns
// of its own half, so neither overwrites columns the other still reads, and the
// MMAs read K-steps 0-3 from column 0 and 4-7 from column 64 of the region.
//
// Masking is a select; rows of Q, dO (dK/dV kernel) and K (dQ kernel) past the
// sequence are zeroed in shared memory up to the 16-row MMA step before they
// enter a contraction over that axis (pad rows may hold NaN and 0 * NaN = NaN).
// Every mbarrier wait is bounded; on expiry THD_DEV_WAIT_TIMEOUT is set, all roles
// stop, loads and MMAs in flight drain and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_launch.h"

namespace thd {

namespace {

using tc::kWaitLimitNs;
using tc::pack2;
using tc::Sync;
using tc_host::encode_view;

constexpr int BT = 128;            // rows per tile on either axis (MMA M and N, TMEM lanes)
constexpr int kThreadsBw = 384;
constexpr int kRegsSoftmax = 184;
constexpr int kRegsControl = 136;
static_assert(2 * kRegsSoftmax + kRegsControl <= 3 * 168, "register split exceeds the launch budget");
constexpr int kAllocWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kIssueWarp = 10;

enum : int {
  B_IN_FULL = 0,       // per-unit operands landed (dQ: Q, dO; dK/dV: K, V)
  B_IN_EMPTY = 1,      // per-unit operands no longer read by MMAs
  B_S_FULL = 2,        // S (or S^T) in TMEM
  B_P_DONE = 3,        // softmax finished its P phase (dQ: S read; dK/dV: P^T stored)
  B_DP_FULL = 4,       // dP (or dP^T) in TMEM
  B_DS_DONE = 5,       // dS (or dS^T) stored in TMEM
  B_ACC_FULL = 6,      // the unit's accumulators are final
  B_ACC_READ = 7,      // the epilogue read them
  B_SCHED_FULL = 8,    // two unit-info slots
  B_SCHED_EMPTY = 10,
  B_FINAL = 12,
  B_RING = 13          // kStages "full" then kStages "empty"
};

template <int D, bool KEYS>
struct BwCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = BT * D * 2;
  static constexpr int kStages = KEYS ? (D == 128 ? 4 : 10) : (D == 128 ? 5 : 10);
  static constexpr int kLdBytes = KEYS ? BT * 8 : 0;      // (LSE2, D) of a query tile, per stage
  static constexpr int kOffFixed = 0;                     // two per-unit tiles
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffLd = kOffRing + kStages * kTileBytes;
  static constexpr int kOffBar = kOffLd + kStages * kLdBytes;
  static constexpr int kNumBars = B_RING + 2 * kStages;
  static constexpr int kOffInfo = kOffBar + kNumBars * 8;
  static constexpr int kOffMisc = kOffInfo + 2 * 80;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kColS = 0;
  static constexpr int kColDP = 128;
  static constexpr int kColAcc = 256;
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory");
  static_assert(kColAcc + (KEYS ? 2 : 1) * D <= 512, "TMEM columns");
};

struct BwUnit {
  uint32_t w;          // work id; >= num_tiles: no more work
  int32_t b, first;    // sequence; first query row (dQ) or first key (dK/dV) of the tile
  int32_t h, g;        // query head (dQ; dK/dV: first head of the kv group), kv head
  int32_t len_q, len_k, shift, lo_shift;
  int32_t off_q, off_k, off_v, off_o;
  int32_t n_valid;     // valid rows (dQ) / keys (dK/dV) of the tile
  int32_t t_lo;        // first KV tile (dQ) / first query tile (dK/dV)
  int32_t n_t;         // KV tiles (dQ) / query tiles per head (dK/dV)
  int32_t n_steps;     // dQ: n_t; dK/dV: query tiles x heads of the kv group, over every member
  int32_t pb;          // pair_base_q[b]: (LSE2, D) block of the sequence's first query tile
  int32_t n_mem;       // dK/dV: sequences of the key group (b, b + 1, ...); 1 for dQ
  int32_t pad;
};
static_assert(sizeof(BwUnit) == 80, "BwUnit is 80 bytes");

__device__ __forceinline__ BwUnit empty_unit(uint32_t w) {
  BwUnit u;
  u.w = w;
  u.b = u.first = u.h = u.g = 0;
  u.len_q = u.len_k = u.shift = u.lo_shift = 0;
  u.off_q = u.off_k = u.off_v = u.off_o = 0;
  u.n_valid = u.t_lo = u.n_t = u.n_steps = u.pb = 0;
  u.n_mem = 1;
  u.pad = 0;
  return u;
}

__device__ __forceinline__ void fill_seq(BwUnit& u, const SeqMeta& m) {
  u.len_q = m.len_q; u.len_k = m.len_k; u.shift = m.shift; u.lo_shift = m.lo_shift;
  u.off_q = m.off_q; u.off_k = m.off_k; u.off_v = m.off_v; u.off_o = m.off_o;
}

// dQ unit: rows [row0, row0 + 128) of one query head; KV tiles from the first
// row's lowest visible key to the last row's highest
__device__ __forceinline__ BwUnit make_unit_dq(const BwdParams& p, uint32_t w, uint32_t num_tiles) {
  BwUnit u = empty_unit(w);
  if (w >= num_tiles) return u;
  int pair, head;
  work_to_unit(p.header_q, w, p.h_q, p.h_kv, pair, head);
  const PairRec pr = p.pairs_q[pair];
  const SeqMeta m = p.meta[pr.b];
  u.b = pr.b; u.first = pr.row0; u.h = head; u.g = head / (p.h_q / p.h_kv);
  fill_seq(u, m);
  const int rows = max(0, min(BT, m.len_q - pr.row0));
  u.n_valid = rows;
  int n = 0, first = 0;
  if (rows > 0) {
    const int64_t kmax = min64((int64_t)m.len_k, (int64_t)pr.row0 + rows - 1 + m.shift + 1);
    const int end = kmax > 0 ? (int)((kmax + BT - 1) / BT) : 0;
    first = (int)(max64(0, (int64_t)pr.row0 + m.lo_shift) / BT);
    n = max(0, end - first);
  }
  u.t_lo = first; u.n_t = n; u.n_steps = n;
  u.pb = p.pair_base_q[pr.b];
  return u;
}

// query tiles [t0, t0 + n) of sequence m that see any key of [k0, k0 + 128):
// key j (< len_k) is seen by rows j - shift <= i <= j - lo_shift
__device__ __forceinline__ void key_block_tiles(const SeqMeta& m, int k0, int& t0, int& n) {
  t0 = 0;
  n = 0;
  const int keys = max(0, min(BT, m.len_k - k0));
  if (m.bad != 0 || keys == 0) return;
  const int64_t i_lo = max64(0, (int64_t)k0 - m.shift);
  const int64_t i_hi = min64((int64_t)m.len_q, (int64_t)k0 + keys - 1 - m.lo_shift + 1);
  if (i_hi > i_lo) {
    t0 = (int)(i_lo / BT);
    n = (int)((i_hi + BT - 1) / BT) - t0;
  }
}

// dK/dV unit: keys [k0, k0 + 128) of one kv head of a key group (the consecutive
// sequences b .. b + n_mem - 1 that read the same K/V rows; usually one); for every
// member and every query head of the kv group, the member's query tiles that see
// those keys. The gradients of all of them accumulate in the unit's TMEM.
__device__ __forceinline__ BwUnit make_unit_dkdv(const BwdParams& p, uint32_t w, uint32_t num_tiles) {
  BwUnit u = empty_unit(w);
  if (w >= num_tiles) return u;
  int pair, g;
  work_to_unit(p.header_k, w, p.h_kv, p.h_kv, pair, g);
  const PairRec pr = p.pairs_k[pair];
  const SeqMeta m = p.meta[pr.b];
  const int group = p.h_q / p.h_kv;
  u.b = pr.b; u.first = pr.row0; u.g = g; u.h = g * group;
  fill_seq(u, m);
  u.n_mem = max(1, m.group_n);
  u.n_valid = max(0, min(BT, m.group_len_k - pr.row0));
  // a lone sequence (the common case) keeps its tiles and pair base in the unit, so
  // the roles walk its steps without reading its metadata again
  int steps = 0;
  key_block_tiles(m, pr.row0, u.t_lo, u.n_t);
  steps = u.n_t * group;
  for (int e = pr.b + 1; e < pr.b + u.n_mem; ++e) {
    int t0, n;
    key_block_tiles(p.meta[e], pr.row0, t0, n);
    steps += n * group;
  }
  u.n_steps = steps;
  u.pb = p.pair_base_q[pr.b];
  return u;
}

// Walks the steps of a dK/dV unit in order: member by member, then query head,
// then query tile. Every role of the kernel walks the same sequence of steps; a
// member's fields are set once per member (`fresh` marks its first step), from the
// unit itself for its first member and from the metadata for the others.
struct StepCursor {
  int e, e_end;        // current member, end of the group
  int t0, t_end;       // the member's query tiles [t0, t_end)
  int hh;              // query head offset inside the kv group
  int h, t;            // query head and query tile of the current step
  int pb;              // pair_base_q of the member
  int len_q, len_k, shift, lo_shift, off_q, off_o;
  bool fresh;          // this step is the member's first
  __device__ __forceinline__ void begin(const BwUnit& u, int group) {
    e = u.b - 1;
    e_end = u.b + u.n_mem;
    t = t_end = 0;
    hh = group - 1;
  }
  // move to the next step (call once before each step of the unit)
  __device__ __forceinline__ void next(const BwdParams& p, const BwUnit& u, int group) {
    fresh = false;
    if (t + 1 < t_end) {
      ++t;
    } else if (hh + 1 < group) {
      ++hh;
      t = t0;
    } else {
      int nt = 0;
      while (nt == 0 && e + 1 < e_end) {
        ++e;
        if (e == u.b) {
          t0 = u.t_lo; nt = u.n_t; pb = u.pb;
          len_q = u.len_q; len_k = u.len_k; shift = u.shift; lo_shift = u.lo_shift;
          off_q = u.off_q; off_o = u.off_o;
        } else {
          const SeqMeta m = p.meta[e];
          key_block_tiles(m, u.first, t0, nt);
          pb = p.pair_base_q[e];
          len_q = m.len_q; len_k = m.len_k; shift = m.shift; lo_shift = m.lo_shift;
          off_q = m.off_q; off_o = m.off_o;
        }
      }
      t_end = t0 + nt;
      t = t0;
      hh = 0;
      fresh = true;
    }
    h = u.h + hh;
  }
};

template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t v, float& lo, float& hi) {
  if constexpr (BF16) {
    lo = __uint_as_float(v << 16);
    hi = __uint_as_float(v & 0xffff0000u);
  } else {
    const __half2 h = *reinterpret_cast<const __half2*>(&v);
    const float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
  }
}

// A operand of the 16-key (or 16-row) step kk of a TMEM-A MMA: each softmax
// warpgroup stored its 64 values packed in the first 32 columns of its half
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

__device__ __forceinline__ uint64_t kmajor_off(int kk) {
  return (uint64_t)((((kk >> 2) * BT * 128) + (kk & 3) * 32) >> 4);
}

struct Ring {
  int stages;
  __device__ __forceinline__ int stage(uint32_t fill) const { return (int)(fill % (uint32_t)stages); }
  __device__ __forceinline__ uint32_t phase(uint32_t fill) const { return (fill / (uint32_t)stages) & 1u; }
};

// barrier setup, TMEM allocation; returns the TMEM base
template <int S>
__device__ __forceinline__ void init_barriers(const Sync& sy) {
  ptx::mbar_init(sy.bar(B_IN_FULL), 1);
  ptx::mbar_init(sy.bar(B_IN_EMPTY), 1);
  ptx::mbar_init(sy.bar(B_S_FULL), 1);
  ptx::mbar_init(sy.bar(B_P_DONE), 8);
  ptx::mbar_init(sy.bar(B_DP_FULL), 1);
  ptx::mbar_init(sy.bar(B_DS_DONE), 8);
  ptx::mbar_init(sy.bar(B_ACC_FULL), 1);
  ptx::mbar_init(sy.bar(B_ACC_READ), 8);
  for (int t = 0; t < 2; ++t) {
    ptx::mbar_init(sy.bar(B_SCHED_FULL + t), 1);
    ptx::mbar_init(sy.bar(B_SCHED_EMPTY + t), 9);   // 8 softmax warps + the issuing thread
  }
  ptx::mbar_init(sy.bar(B_FINAL), 1);
  for (int s = 0; s < S; ++s) {
    ptx::mbar_init(sy.bar(B_RING + s), 1);
    ptx::mbar_init(sy.bar(B_RING + S + s), 1);
  }
}

// after an abort the producer waits (bounded) for the loads it issued
template <int S>
__device__ __forceinline__ void drain_loads(const Sync& sy, uint32_t fill, uint32_t in_uses) {
  for (int s = 0; s < S; ++s) {
    if (fill > (uint32_t)s) {
      const uint32_t last = (fill - 1 - (uint32_t)s) / S * S + (uint32_t)s;
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(sy.bar(B_RING + s), (last / S) & 1u) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
  if (in_uses > 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(sy.bar(B_IN_FULL), (in_uses - 1) & 1u) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  }
}

__device__ __forceinline__ void drain_mmas(const Sync& sy) {
  ptx::tc_commit(sy.bar(B_FINAL));
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(sy.bar(B_FINAL), 0) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// zero rows [valid, valid + n) of a 128-row tile (whole 128-byte rows: swizzle-agnostic)
template <int HALVES>
__device__ __forceinline__ void zero_rows(uint8_t* tile, int valid, int n) {
  for (int hf = 0; hf < HALVES; ++hf)
    for (int idx = 0; idx < n * 8; ++idx)
      *reinterpret_cast<uint4*>(tile + hf * BT * 128 + valid * 128 + idx * 16) = make_uint4(0, 0, 0, 0);
}

// ============================================================================ dQ
template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kThreadsBw, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using C = BwCfg<D, false>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  BwUnit* info = reinterpret_cast<BwUnit*>(smem + C::kOffInfo);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);
  // short spins before the sleep-hinted waits: a softmax warp that polls long
  // takes issue slots from the warps (and the issuing thread) on its sub-partition
  const Sync sy{sbase + (uint32_t)C::kOffBar, abort_flag, p.status, 4};
  const Ring ring{C::kStages};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t num_tiles = p.header_q[kHdrNumTiles];

  if (threadIdx.x == 0) {
    init_barriers<C::kStages>(sy);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
  }
  if (warp == kAllocWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kRegsControl>();
    if (warp == kTmaWarp && lane == 0) {
      // ------------------------------------------------ scheduler + TMA producer
      uint32_t in_uses = 0, fill = 0;
      for (uint32_t it = 0;; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_EMPTY + slot, ((it >> 1) & 1u) ^ 1u)) break;
        const uint32_t w = atomicAdd(p.counter_q, 1u);
        const BwUnit u = make_unit_dq(p, w, num_tiles);
        info[slot] = u;
        ptx::mbar_arrive(sy.bar(B_SCHED_FULL + slot));
        if (w >= num_tiles) break;
        if (u.n_steps == 0) continue;
        if (!sy.wait(B_IN_EMPTY, (in_uses & 1u) ^ 1u)) break;
        ++in_uses;
        ptx::mbar_arrive_expect_tx(sy.bar(B_IN_FULL), 2 * C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          ptx::tma_load_3d(sbase + C::kOffFixed + hf * BT * 128, &tm_q, sy.bar(B_IN_FULL), hf * 64, u.h,
                           u.off_q + u.first);
          ptx::tma_load_3d(sbase + C::kOffFixed + C::kTileBytes + hf * BT * 128, &tm_do, sy.bar(B_IN_FULL),
                           hf * 64, u.h, u.off_o + u.first);
        }
        bool ok = true;
        for (int j = 0; j < u.n_steps && ok; ++j) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int st = ring.stage(fill);
            if (!(ok = sy.wait(B_RING + C::kStages + st, ring.phase(fill) ^ 1u))) break;
            ++fill;
            ptx::mbar_arrive_expect_tx(sy.bar(B_RING + st), C::kTileBytes);
            const void* map = kv == 0 ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
            const int row = (kv == 0 ? u.off_k : u.off_v) + (u.t_lo + j) * BT;
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
              ptx::tma_load_3d(sbase + C::kOffRing + st * C::kTileBytes + hf * BT * 128, map, sy.bar(B_RING + st),
                               hf * 64, u.g, row);
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) drain_loads<C::kStages>(sy, fill, in_uses);
    }
    if (warp == kIssueWarp && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      constexpr uint32_t kIdescSq = ptx::idesc_f16(BF16, BT, BT, false);
      constexpr uint32_t kIdescAcc = ptx::idesc_f16(BF16, BT, D, true);
      const uint64_t dq_a = ptx::sdesc_sw128(sbase + C::kOffFixed, 16, 1024);
      const uint64_t ddo_a = ptx::sdesc_sw128(sbase + C::kOffFixed + C::kTileBytes, 16, 1024);
      const uint64_t dring_k = ptx::sdesc_sw128(sbase + C::kOffRing, 16, 1024);
      const uint64_t dring_mn = ptx::sdesc_sw128(sbase + C::kOffRing, BT * 128, 1024);
      const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tAcc = tmem + C::kColAcc;
      auto issue_sq = [&](uint32_t dst, uint64_t a, int st) {
        const uint64_t b = dring_k + (uint64_t)((st * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) ptx::mma_ss(dst, a + kmajor_off(kk), b + kmajor_off(kk), kIdescSq, kk > 0);
      };
      auto issue_dq = [&](int st, bool acc, int nk) {
        const uint64_t b = dring_mn + (uint64_t)((st * C::kTileBytes) >> 4);
        for (int kk = 0; kk < nk; ++kk)
          ptx::mma_ts(tAcc, tDP + packed_col(kk), b + (uint64_t)(kk * 128), kIdescAcc, (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t in_uses = 0, p_waits = 0, ds_waits = 0, acc_reads_seen = 0, acc_read_waits = 0, base = 0;
      bool issued_any = false, ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
        const BwUnit u = info[slot];
        ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
        if (u.w >= num_tiles) break;
        const int n = u.n_steps;
        if (n == 0) continue;
        const uint32_t k0f = base, v0f = base + 1;
        ok = sy.wait(B_IN_FULL, (in_uses++) & 1u) && sy.wait(B_RING + ring.stage(k0f), ring.phase(k0f));
        if (!ok) break;
        ptx::tc_fence_after();
        issue_sq(tS, dq_a, ring.stage(k0f));
        ptx::tc_commit(sy.bar(B_S_FULL));
        if (!(ok = sy.wait(B_RING + ring.stage(v0f), ring.phase(v0f)))) break;
        ptx::tc_fence_after();
        issue_sq(tDP, ddo_a, ring.stage(v0f));
        ptx::tc_commit(sy.bar(B_DP_FULL));
        ptx::tc_commit(sy.bar(B_RING + C::kStages + ring.stage(v0f)));
        if (n == 1) ptx::tc_commit(sy.bar(B_IN_EMPTY));
        issued_any = true;
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t kf = base + 2u * j, kf1 = kf + 2u, vf1 = kf + 3u;
          // S(j) read by the softmax: S(j+1) may overwrite it
          if (!(ok = sy.wait(B_P_DONE, (p_waits++) & 1u))) break;
          if (j + 1 < n) {
            if (!(ok = sy.wait(B_RING + ring.stage(kf1), ring.phase(kf1)))) break;
            ptx::tc_fence_after();
            issue_sq(tS, dq_a, ring.stage(kf1));
            ptx::tc_commit(sy.bar(B_S_FULL));
          }
          if (!(ok = sy.wait(B_DS_DONE, (ds_waits++) & 1u))) break;
          while (ok && j == 0 && acc_read_waits < acc_reads_seen) ok = sy.wait(B_ACC_READ, (acc_read_waits++) & 1u);
          if (!ok) break;
          // keys of this tile past len_k: dQ runs over ceil(valid/16) steps of 16 keys
          // and the at most 15 K rows between are zeroed (S(j) has completed)
          int nk = BT / 16;
          const int jj = u.t_lo + j;
          if ((jj + 1) * BT > u.len_k) {
            const int valid = u.len_k - jj * BT;
            nk = (valid + 15) >> 4;
            if (nk * 16 > valid) {
              zero_rows<C::kHalves>(smem + C::kOffRing + ring.stage(kf) * C::kTileBytes, valid, nk * 16 - valid);
              ptx::fence_proxy_async_smem();
            }
          }
          ptx::tc_fence_after();
          issue_dq(ring.stage(kf), j > 0, nk);
          ptx::tc_commit(sy.bar(B_RING + C::kStages + ring.stage(kf)));
          if (j + 1 < n) {
            if (!(ok = sy.wait(B_RING + ring.stage(vf1), ring.phase(vf1)))) break;
            ptx::tc_fence_after();
            issue_sq(tDP, ddo_a, ring.stage(vf1));
            ptx::tc_commit(sy.bar(B_DP_FULL));
            ptx::tc_commit(sy.bar(B_RING + C::kStages + ring.stage(vf1)));
            if (j + 2 == n) ptx::tc_commit(sy.bar(B_IN_EMPTY));
          } else {
            ptx::tc_commit(sy.bar(B_ACC_FULL));
          }
        }
        base += 2u * (uint32_t)n;
        ++acc_reads_seen;
      }
      if (issued_any) drain_mmas(sy);
    }
    __syncwarp();
  } else {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    // ----------------------------------------------- softmax: row = TMEM lane, 64 keys
    const int wg = warp >> 2;                    // which half of the 128 keys / D columns
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_bits = (uint32_t)((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_bits + (uint32_t)(C::kColS + wg * 64);
    const uint32_t tDP = tmem + lane_bits + (uint32_t)(C::kColDP + wg * 64);
    const uint32_t tAcc = tmem + lane_bits + (uint32_t)(C::kColAcc + wg * (D / 2));
    const float sl2 = p.scale_log2;
    T* __restrict__ DQ = static_cast<T*>(p.dq);
    auto warp_arrive = [&](int b) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(b));
    };
    uint32_t s_cnt = 0, dp_cnt = 0, acc_cnt = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = (int)(it & 1u);
      if (!sy.wait_warp(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
      const BwUnit u = info[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
      if (u.w >= num_tiles) break;
      const int r = u.first + row;
      const bool live = row < u.n_valid;
      float lse2 = INFINITY, dsum = 0.f;
      if (live) {
        const float2 ld = p.ld[((int64_t)(u.pb + u.first / BT) * p.h_q + u.h) * BT + row];
        lse2 = ld.x;
        dsum = ld.y;
      }
      const int kmax_row = live ? (int)max64(0, min64((int64_t)u.len_k, (int64_t)r + u.shift + 1)) : 0;
      const int kmin_row = WIN ? (int)max64(0, min64((int64_t)u.len_k, (int64_t)r + u.lo_shift)) : 0;
      bool ok = true;
      for (int j = 0; j < u.n_steps; ++j) {
        if (!(ok = sy.wait_warp(B_S_FULL, (s_cnt++) & 1u))) break;
        ptx::tc_fence_after();
        uint32_t s[2][32];
        ptx::tmem_ld32(tS, s[0]);
        ptx::tmem_ld32(tS + 32, s[1]);
        ptx::tmem_wait_ld(s[0]);
        ptx::tmem_wait_ld(s[1]);
        warp_arrive(B_P_DONE);                   // S read: the next S may overwrite it
        const int c0 = (u.t_lo + j) * BT + wg * 64;   // key of column 0 of this half
        const int lim = kmax_row - c0, lim_lo = kmin_row - c0;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0 = ptx::ex2(fmaf(__uint_as_float(s[c >> 5][c & 31]), sl2, -lse2));
          float x1 = ptx::ex2(fmaf(__uint_as_float(s[c >> 5][(c + 1) & 31]), sl2, -lse2));
          if (c >= lim || (WIN && c < lim_lo)) x0 = 0.f;
          if (c + 1 >= lim || (WIN && c + 1 < lim_lo)) x1 = 0.f;
          pk[c >> 1] = pack2<BF16>(x0, x1);
        }
        if (!(ok = sy.wait_warp(B_DP_FULL, (dp_cnt++) & 1u))) break;
        ptx::tc_fence_after();
        ptx::tmem_ld32(tDP, s[0]);
        ptx::tmem_ld32(tDP + 32, s[1]);
        ptx::tmem_wait_ld(s[0]);
        ptx::tmem_wait_ld(s[1]);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float p0, p1;
          unpack2<BF16>(pk[c >> 1], p0, p1);
          const float d0 = p0 > 0.f ? p0 * (__uint_as_float(s[c >> 5][c & 31]) - dsum) : 0.f;
          const float d1 = p1 > 0.f ? p1 * (__uint_as_float(s[c >> 5][(c + 1) & 31]) - dsum) : 0.f;
          pk[c >> 1] = pack2<BF16>(d0, d1);
        }
        ptx::tmem_st32(tDP, pk);
        ptx::tmem_wait_st();
        warp_arrive(B_DS_DONE);
      }
      if (!ok) break;
      // epilogue: dQ = scale * acc on live rows; rows with no KV tile get 0
      T* qrow = DQ + (int64_t)(u.off_q + r) * p.stride_tok[5] + (int64_t)u.h * p.stride_head[5] + wg * (D / 2);
      if (u.n_steps > 0) {
        if (!sy.wait_warp(B_ACC_FULL, (acc_cnt++) & 1u)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tAcc + 32 * c, o);
          ptx::tmem_wait_ld(o);
          if (live) {
            uint32_t pq[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pq[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * p.scale, __uint_as_float(o[2 * i + 1]) * p.scale);
            uint4* dst = reinterpret_cast<uint4*>(qrow + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(pq[4 * q4], pq[4 * q4 + 1], pq[4 * q4 + 2], pq[4 * q4 + 3]);
          }
        }
        warp_arrive(B_ACC_READ);
      } else if (live) {
        uint4* dst = reinterpret_cast<uint4*>(qrow);
#pragma unroll
        for (int q4 = 0; q4 < D / 16; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kAllocWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dK, dV
template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kThreadsBw, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = BwCfg<D, true>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  BwUnit* info = reinterpret_cast<BwUnit*>(smem + C::kOffInfo);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);
  // short spins before the sleep-hinted waits: a softmax warp that polls long
  // takes issue slots from the warps (and the issuing thread) on its sub-partition
  const Sync sy{sbase + (uint32_t)C::kOffBar, abort_flag, p.status, 4};
  const Ring ring{C::kStages};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t num_tiles = p.header_k[kHdrNumTiles];
  const int group = p.h_q / p.h_kv;   // query heads per kv head

  if (threadIdx.x == 0) {
    init_barriers<C::kStages>(sy);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
  }
  if (warp == kAllocWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kRegsControl>();
    if (warp == kTmaWarp && lane == 0) {
      // ------------------------------------------------ scheduler + TMA producer
      uint32_t in_uses = 0, fill = 0;
      for (uint32_t it = 0;; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_EMPTY + slot, ((it >> 1) & 1u) ^ 1u)) break;
        const uint32_t w = atomicAdd(p.counter_k, 1u);
        const BwUnit u = make_unit_dkdv(p, w, num_tiles);
        info[slot] = u;
        ptx::mbar_arrive(sy.bar(B_SCHED_FULL + slot));
        if (w >= num_tiles) break;
        if (u.n_steps == 0) continue;
        if (!sy.wait(B_IN_EMPTY, (in_uses & 1u) ^ 1u)) break;
        ++in_uses;
        ptx::mbar_arrive_expect_tx(sy.bar(B_IN_FULL), 2 * C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          ptx::tma_load_3d(sbase + C::kOffFixed + hf * BT * 128, &tm_k, sy.bar(B_IN_FULL), hf * 64, u.g,
                           u.off_k + u.first);
          ptx::tma_load_3d(sbase + C::kOffFixed + C::kTileBytes + hf * BT * 128, &tm_v, sy.bar(B_IN_FULL),
                           hf * 64, u.g, u.off_v + u.first);
        }
        bool ok = true;
        StepCursor cur;
        cur.begin(u, group);
        for (int i = 0; i < u.n_steps && ok; ++i) {
          cur.next(p, u, group);
          const int h = cur.h;
          const int t = cur.t;
#pragma unroll
          for (int x = 0; x < 2; ++x) {     // 0: Q_i with its (LSE2, D) block, 1: dO_i
            const int st = ring.stage(fill);
            if (!(ok = sy.wait(B_RING + C::kStages + st, ring.phase(fill) ^ 1u))) break;
            ++fill;
            const uint32_t fb = sy.bar(B_RING + st);
            ptx::mbar_arrive_expect_tx(fb, C::kTileBytes + (x == 0 ? C::kLdBytes : 0));
            const void* map = x == 0 ? static_cast<const void*>(&tm_q) : static_cast<const void*>(&tm_do);
            const int row = (x == 0 ? cur.off_q : cur.off_o) + t * BT;
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
              ptx::tma_load_3d(sbase + C::kOffRing + st * C::kTileBytes + hf * BT * 128, map, fb, hf * 64, h, row);
            if (x == 0)
              ptx::bulk_load(sbase + C::kOffLd + st * C::kLdBytes, p.ld + ((int64_t)(cur.pb + t) * p.h_q + h) * BT,
                             C::kLdBytes, fb);
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) drain_loads<C::kStages>(sy, fill, in_uses);
    }
    if (warp == kIssueWarp && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      constexpr uint32_t kIdescSq = ptx::idesc_f16(BF16, BT, BT, false);
      constexpr uint32_t kIdescAcc = ptx::idesc_f16(BF16, BT, D, true);
      const uint64_t dk_a = ptx::sdesc_sw128(sbase + C::kOffFixed, 16, 1024);
      const uint64_t dv_a = ptx::sdesc_sw128(sbase + C::kOffFixed + C::kTileBytes, 16, 1024);
      const uint64_t dring_k = ptx::sdesc_sw128(sbase + C::kOffRing, 16, 1024);
      const uint64_t dring_mn = ptx::sdesc_sw128(sbase + C::kOffRing, BT * 128, 1024);
      const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP;
      const uint32_t tDV = tmem + C::kColAcc, tDK = tmem + C::kColAcc + D;
      auto issue_sq = [&](uint32_t dst, uint64_t a, int st) {
        const uint64_t b = dring_k + (uint64_t)((st * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) ptx::mma_ss(dst, a + kmajor_off(kk), b + kmajor_off(kk), kIdescSq, kk > 0);
      };
      auto issue_acc = [&](uint32_t dst, uint32_t a_tmem, int st, bool acc, int nk) {
        const uint64_t b = dring_mn + (uint64_t)((st * C::kTileBytes) >> 4);
        for (int kk = 0; kk < nk; ++kk)
          ptx::mma_ts(dst, a_tmem + packed_col(kk), b + (uint64_t)(kk * 128), kIdescAcc, (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t in_uses = 0, p_waits = 0, dp_waits = 0, ds_waits = 0, acc_reads_seen = 0, acc_read_waits = 0;
      uint32_t base = 0;
      bool issued_any = false, ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
        const BwUnit u = info[slot];
        ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
        if (u.w >= num_tiles) break;
        const int n = u.n_steps;
        if (n == 0) continue;
        ok = sy.wait(B_IN_FULL, (in_uses++) & 1u) && sy.wait(B_RING + ring.stage(base), ring.phase(base));
        if (!ok) break;
        ptx::tc_fence_after();
        issue_sq(tS, dk_a, ring.stage(base));
        ptx::tc_commit(sy.bar(B_S_FULL));
        if (!(ok = sy.wait(B_RING + ring.stage(base + 1), ring.phase(base + 1)))) break;
        ptx::tc_fence_after();
        issue_sq(tDP, dv_a, ring.stage(base + 1));
        ptx::tc_commit(sy.bar(B_DP_FULL));
        if (n == 1) ptx::tc_commit(sy.bar(B_IN_EMPTY));
        issued_any = true;
        StepCursor cur;
        cur.begin(u, group);
        for (int i = 0; i < n && ok; ++i) {
          const uint32_t qf = base + 2u * i, of = qf + 1u, qf1 = qf + 2u, of1 = qf + 3u;
          // query rows of this tile past len_q: dV and dK run over ceil(valid/16)
          // steps of 16 rows and the at most 15 rows between are zeroed in Q_i / dO_i
          cur.next(p, u, group);
          const int valid = min(BT, cur.len_q - cur.t * BT);
          const int nk = (valid + 15) >> 4;
          const int zr = nk * 16 - valid;
          if (!(ok = sy.wait(B_P_DONE, (p_waits++) & 1u))) break;
          while (ok && i == 0 && acc_read_waits < acc_reads_seen) ok = sy.wait(B_ACC_READ, (acc_read_waits++) & 1u);
          // dP(i) has read dO_i before its tail rows are cleared (only the last query
          // tile of a sequence has a tail; the phase count advances every step)
          const uint32_t dp_phase = dp_waits++;
          if (zr > 0) ok = ok && sy.wait(B_DP_FULL, dp_phase & 1u);
          if (!ok) break;
          if (zr > 0) {
            zero_rows<C::kHalves>(smem + C::kOffRing + ring.stage(of) * C::kTileBytes, valid, zr);
            ptx::fence_proxy_async_smem();
          }
          ptx::tc_fence_after();
          issue_acc(tDV, tS, ring.stage(of), i > 0, nk);
          ptx::tc_commit(sy.bar(B_RING + C::kStages + ring.stage(of)));
          if (i + 1 < n) {
            if (!(ok = sy.wait(B_RING + ring.stage(qf1), ring.phase(qf1)))) break;
            ptx::tc_fence_after();
            issue_sq(tS, dk_a, ring.stage(qf1));
            ptx::tc_commit(sy.bar(B_S_FULL));
          }
          if (!(ok = sy.wait(B_DS_DONE, (ds_waits++) & 1u))) break;
          if (zr > 0) {
            zero_rows<C::kHalves>(smem + C::kOffRing + ring.stage(qf) * C::kTileBytes, valid, zr);
            ptx::fence_proxy_async_smem();
          }
          ptx::tc_fence_after();
          issue_acc(tDK, tDP, ring.stage(qf), i > 0, nk);
          ptx::tc_commit(sy.bar(B_RING + C::kStages + ring.stage(qf)));
          if (i + 1 < n) {
            if (!(ok = sy.wait(B_RING + ring.stage(of1), ring.phase(of1)))) break;
            ptx::tc_fence_after();
            issue_sq(tDP, dv_a, ring.stage(of1));
            ptx::tc_commit(sy.bar(B_DP_FULL));
            if (i + 2 == n) ptx::tc_commit(sy.bar(B_IN_EMPTY));
          } else {
            ptx::tc_commit(sy.bar(B_ACC_FULL));
          }
        }
        base += 2u * (uint32_t)n;
        ++acc_reads_seen;
      }
      if (issued_any) drain_mmas(sy);
    }
    __syncwarp();
  } else {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    // ----------------------------------------- softmax: key = TMEM lane, 64 queries
    const int wg = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_bits = (uint32_t)((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_bits + (uint32_t)(C::kColS + wg * 64);
    const uint32_t tDP = tmem + lane_bits + (uint32_t)(C::kColDP + wg * 64);
    const uint32_t tDV = tmem + lane_bits + (uint32_t)(C::kColAcc + wg * (D / 2));
    const uint32_t tDK = tDV + D;
    const float sl2 = p.scale_log2;
    T* __restrict__ DK = static_cast<T*>(p.dk);
    T* __restrict__ DV = static_cast<T*>(p.dv);
    auto warp_arrive = [&](int b) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(b));
    };
    uint32_t s_cnt = 0, dp_cnt = 0, acc_cnt = 0, base = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = (int)(it & 1u);
      if (!sy.wait_warp(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
      const BwUnit u = info[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
      if (u.w >= num_tiles) break;
      const int64_t j = (int64_t)u.first + row;     // key inside the sequence
      const bool live = row < u.n_valid;            // key of the group
      bool ok = true;
      StepCursor cur;
      cur.begin(u, group);
      bool live_m = false;
      int64_t i_min = 0, i_end = 0;
      for (int i = 0; i < u.n_steps; ++i) {
        const uint32_t qf = base + 2u * i;
        cur.next(p, u, group);
        if (cur.fresh) {
          // visible query rows of this key for the step's member: j < len_k and
          // j - shift <= i <= j - lo_shift, i < len_q
          live_m = live && j < cur.len_k;
          i_min = j - cur.shift;
          i_end = min64((int64_t)cur.len_q, j - (int64_t)cur.lo_shift + 1);
        }
        const int t = cur.t;
        const int64_t cb = (int64_t)t * BT + wg * 64;     // query row of column 0 of this half
        const int c_lo = live_m ? (int)max64(0, min64(64, i_min - cb)) : 64;
        const int c_hi = live_m ? (int)max64(0, min64(64, i_end - cb)) : 0;
        const float2* lds = reinterpret_cast<const float2*>(smem + C::kOffLd + ring.stage(qf) * C::kLdBytes) + wg * 64;
        if (!(ok = sy.wait_warp(B_S_FULL, (s_cnt++) & 1u))) break;
        // the (LSE2, D) block arrived with Q_i on this stage's barrier
        if (!(ok = sy.wait_warp(B_RING + ring.stage(qf), ring.phase(qf)))) break;
        ptx::tc_fence_after();
        uint32_t s[2][32];
        ptx::tmem_ld32(tS, s[0]);
        ptx::tmem_ld32(tS + 32, s[1]);
        ptx::tmem_wait_ld(s[0]);
        ptx::tmem_wait_ld(s[1]);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float x0 = ptx::ex2(fmaf(__uint_as_float(s[c >> 5][c & 31]), sl2, -lds[c].x));
          float x1 = ptx::ex2(fmaf(__uint_as_float(s[c >> 5][(c + 1) & 31]), sl2, -lds[c + 1].x));
          if (c < c_lo || c >= c_hi) x0 = 0.f;
          if (c + 1 < c_lo || c + 1 >= c_hi) x1 = 0.f;
          pk[c >> 1] = pack2<BF16>(x0, x1);
        }
        ptx::tmem_st32(tS, pk);
        ptx::tmem_wait_st();
        warp_arrive(B_P_DONE);
        if (!(ok = sy.wait_warp(B_DP_FULL, (dp_cnt++) & 1u))) break;
        ptx::tc_fence_after();
        ptx::tmem_ld32(tDP, s[0]);
        ptx::tmem_ld32(tDP + 32, s[1]);
        ptx::tmem_wait_ld(s[0]);
        ptx::tmem_wait_ld(s[1]);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float p0, p1;
          unpack2<BF16>(pk[c >> 1], p0, p1);
          const float d0 = p0 > 0.f ? p0 * (__uint_as_float(s[c >> 5][c & 31]) - lds[c].y) : 0.f;
          const float d1 = p1 > 0.f ? p1 * (__uint_as_float(s[c >> 5][(c + 1) & 31]) - lds[c + 1].y) : 0.f;
          pk[c >> 1] = pack2<BF16>(d0, d1);
        }
        ptx::tmem_st32(tDP, pk);
        ptx::tmem_wait_st();
        warp_arrive(B_DS_DONE);
      }
      if (!ok) break;
      base += 2u * (uint32_t)u.n_steps;
      T* krow = DK + (int64_t)(u.off_k + j) * p.stride_tok[6] + (int64_t)u.g * p.stride_head[6] + wg * (D / 2);
      T* vrow = DV + (int64_t)(u.off_v + j) * p.stride_tok[7] + (int64_t)u.g * p.stride_head[7] + wg * (D / 2);
      if (u.n_steps > 0) {
        if (!sy.wait_warp(B_ACC_FULL, (acc_cnt++) & 1u)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tDV + 32 * c, o);
          ptx::tmem_wait_ld(o);
          if (live) {
            uint32_t pq[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) pq[x] = pack2<BF16>(__uint_as_float(o[2 * x]), __uint_as_float(o[2 * x + 1]));
            uint4* dst = reinterpret_cast<uint4*>(vrow + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(pq[4 * q4], pq[4 * q4 + 1], pq[4 * q4 + 2], pq[4 * q4 + 3]);
          }
          ptx::tmem_ld32(tDK + 32 * c, o);
          ptx::tmem_wait_ld(o);
          if (live) {
            uint32_t pq[16];
#pragma unroll
            for (int x = 0; x < 16; ++x)
              pq[x] = pack2<BF16>(__uint_as_float(o[2 * x]) * p.scale, __uint_as_float(o[2 * x + 1]) * p.scale);
            uint4* dst = reinterpret_cast<uint4*>(krow + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(pq[4 * q4], pq[4 * q4 + 1], pq[4 * q4 + 2], pq[4 * q4 + 3]);
          }
        }
        warp_arrive(B_ACC_READ);
      } else if (live) {
#pragma unroll
        for (int q4 = 0; q4 < D / 16; ++q4) {
          reinterpret_cast<uint4*>(krow)[q4] = make_uint4(0, 0, 0, 0);
          reinterpret_cast<uint4*>(vrow)[q4] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kAllocWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool WIN>
cudaError_t launch_bwd_impl(const BwdParams& p, const thd_attn_desc_t& desc, const int64_t g_cap[4],
                            const int64_t g_stok[4], const int64_t g_shead[4], int max_q, int max_k, int num_sms,
                            cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_view(&tq, p.q, BF16, D, desc.h_q, desc.cap_rows[0], desc.stride_head[0], desc.stride_tok[0]) ||
      !encode_view(&tk, p.k, BF16, D, desc.h_kv, desc.cap_rows[1], desc.stride_head[1], desc.stride_tok[1]) ||
      !encode_view(&tv, p.v, BF16, D, desc.h_kv, desc.cap_rows[2], desc.stride_head[2], desc.stride_tok[2]) ||
      !encode_view(&tdo, p.d_o, BF16, D, desc.h_q, g_cap[0], g_shead[0], g_stok[0]))
    return cudaErrorNotSupported;
  {
    using C = BwCfg<D, false>;
    const int smem = C::kSmemBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D, BF16, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)max64(1, min64((int64_t)num_sms, (int64_t)max_q * desc.h_q));
    bwd_dq_tc_kernel<D, BF16, WIN><<<grid, kThreadsBw, smem, stream>>>(tq, tk, tv, tdo, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    using C = BwCfg<D, true>;
    const int smem = C::kSmemBytes + 1024;
    cudaError_t e =
        cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D, BF16, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int grid = (int)max64(1, min64((int64_t)num_sms, (int64_t)max_k * desc.h_kv));
    bwd_dkdv_tc_kernel<D, BF16, WIN><<<grid, kThreadsBw, smem, stream>>>(tq, tk, tv, tdo, p);
    return cudaGetLastError();
  }
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdParams& p, const thd_attn_desc_t& desc, const int64_t g_cap[4],
                          const int64_t g_stok[4], const int64_t g_shead[4], int max_q, int max_k, int num_sms,
                          cudaStream_t stream) {
  const bool bf16 = desc.dtype == THD_BF16;
  const bool win = p.has_window != 0;
#define THD_BW_LAUNCH(D_, B_)                                                                               \
  return win ? launch_bwd_impl<D_, B_, true>(p, desc, g_cap, g_stok, g_shead, max_q, max_k, num_sms, stream) \
             : launch_bwd_impl<D_, B_, false>(p, desc, g_cap, g_stok, g_shead, max_q, max_k, num_sms, stream)
  if (desc.d == 128) {
    if (bf16) THD_BW_LAUNCH(128, true);
    THD_BW_LAUNCH(128, false);
  }
  if (desc.d == 64) {
    if (bf16) THD_BW_LAUNCH(64, true);
    THD_BW_LAUNCH(64, false);
  }
#undef THD_BW_LAUNCH
  return cudaErrorNotSupported;
}

}  // namespace thd
