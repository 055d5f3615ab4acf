// Tensor-core forward kernel for sm_103a: TMA-staged Q/K/V tiles, tcgen05.mma
// into TMEM for S = Q K^T and O += P V, online softmax in fp32 by warps that own
// one TMEM lane (query row) each.
//
// Work unit: 256 query rows (two 128-row sub-tiles) of one sequence and one query
// head, claimed from the workspace tile counter by a persistent CTA
// (cudnn-frontend PR #462, "Root cause": tile_id = atomicAdd(counter, 1); retire
// once tile_id >= num_tiles). Rows are addressed through the caller's ragged
// offsets as TMA coordinates over the whole [rows, heads, d] view
// (cuDNN-frontend issue "THD lowering never reads the bound ragged offsets",
// "Concrete failure": the per-sequence offset enters as a TMA row coordinate).
//
// Warp roles (384 threads = 3 warpgroups, one CTA per SM):
//   warps 0-3   softmax of sub-tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax of sub-tile 1
//   warp  8     TMEM allocation / release
//   warp  9     scheduler + TMA producer (one thread)
//   warp  10    MMA issue (one thread); warp 11 idle
// The third warpgroup gives registers back (setmaxnreg) so each softmax thread can
// hold a full 128-column row of S without spilling.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D, 256+2D).
// P (bf16/fp16, two per 32-bit column) overwrites the first 64 columns of its S.
// Shared memory: Q0, Q1 and a ring of K/V tiles; at d = 128 each ring slot has its
// own full/empty mbarrier pair, at d = 64 one pair covers the tiles V_j and K_{j+1}
// that one tile's MMA batches consume (Cfg::kGroupKV).
//
// The issuing thread orders MMAs PV0(j), QK0(j+1), PV1(j), QK1(j+1): the two
// sub-tiles alternate on the tensor core, and each softmax runs while the other
// sub-tile's MMAs execute. The commit that signals S_t(j+1) also covers PV_t(j),
// so O_t can be rescaled in place as soon as S_t(j+1) is ready.
//
// Masking is a select (s = visible ? s : -inf), never an added bias, and the V
// rows of the last KV tile past len_k are zeroed in shared memory before PV:
// pad rows may hold NaN (the context-parallel padding case of the cuDNN-frontend
// issue has "no initialization guarantee", and 0 * NaN = NaN). Only rows
// r < len_q are stored, so pad rows of O and Stats are never written.
//
// Every mbarrier wait is bounded (4 s of %globaltimer); on expiry the kernel sets
// THD_DEV_WAIT_TIMEOUT in the status word, all roles leave their loops, MMAs in
// flight are drained and TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_launch.h"

namespace thd {

// Optional timeline of the kernel's hand-offs, compiled only with -DTHD_FWD_TRACE
// (the library is built without it; ragged_varlen_attention_gb300.profiling.fwd_timeline
// builds a traced copy): clock64() stamps of the first unit of each CTA, per KV
// tile j < kTrTiles, for the two softmax warpgroups (role = sub-tile) and the
// MMA-issuing thread (role 2). Softmax events: 0 before the S wait, 1 S ready,
// 2 S in registers, 3 P computed, 4 P stored, 5 arrived. Issuer events: 0 loop top,
// 1 V_j and K_{j+1} ready, 2 / 4 P_0 / P_1 ready, 3 / 5 after batch 0 / 1 and its
// commits, 6 after the stage releases.
#ifdef THD_FWD_TRACE
constexpr int kTrCtas = 160, kTrRoles = 3, kTrTiles = 64, kTrEvents = 8;
__device__ unsigned long long g_fwd_trace[kTrCtas * kTrRoles * kTrTiles * kTrEvents];
__device__ __forceinline__ void trace_stamp(int role, int j, int ev, uint32_t unit_it) {
  if (unit_it == 0 && blockIdx.x < kTrCtas && j >= 0 && j < kTrTiles)
    g_fwd_trace[((blockIdx.x * kTrRoles + role) * kTrTiles + j) * kTrEvents + ev] = clock64();
}
#define THD_TRACE_STAMP(role, j, ev, it) trace_stamp(role, j, ev, it)
// per CTA and unit u < kTrUnits, %globaltimer (ns, one clock for all SMs): 0 unit
// claimed, 1 its loads issued, 2 issuing thread has it, 3 first QK committed, 4 last
// MMA committed, 5 / 6 epilogue of sub-tile 0 / 1 stored, 7 (work id << 32) | KV tiles.
// g_fwd_cta: CTA start (after the prologue) and end.
constexpr int kTrUnits = 16, kTrUEvents = 8;
__device__ unsigned long long g_fwd_units[kTrCtas * kTrUnits * kTrUEvents];
__device__ unsigned long long g_fwd_cta[kTrCtas * 2];
__device__ __forceinline__ void unit_stamp(uint32_t u, int ev, unsigned long long v) {
  if (blockIdx.x < kTrCtas && u < kTrUnits) g_fwd_units[(blockIdx.x * kTrUnits + u) * kTrUEvents + ev] = v;
}
#define THD_UNIT_STAMP(u, ev) unit_stamp(u, ev, ptx::globaltimer_ns())
#define THD_UNIT_INFO(u, v) unit_stamp(u, 7, v)
#define THD_CTA_STAMP(ev) do { if (blockIdx.x < kTrCtas) g_fwd_cta[blockIdx.x * 2 + (ev)] = ptx::globaltimer_ns(); } while (0)
#else
#define THD_TRACE_STAMP(role, j, ev, it) ((void)0)
#define THD_UNIT_STAMP(u, ev) ((void)0)
#define THD_UNIT_INFO(u, v) ((void)0)
#define THD_CTA_STAMP(ev) ((void)0)
#endif

namespace {

using tc::Sync;
using tc::kWaitLimitNs;
using tc::pack2;
using tc_host::encode_view;

constexpr int BM = 128;           // query rows per sub-tile (MMA M, TMEM lanes)
constexpr int BN = 128;           // keys per KV tile
constexpr int kThreadsTC = 384;
// launch budget 168 registers/thread (384 x 168 = 64512); warpgroup 2 (MMA, TMA,
// idle warps) drops to 120 and the two softmax warpgroups rise to 192:
// 128 x (2 x 192 + 120) = 64512, so every increase can be granted (at 184 the
// softmax spilled a few values through the tile loop)
constexpr int kRegsSoftmax = 192;
constexpr int kRegsControl = 120;
static_assert(2 * kRegsSoftmax + kRegsControl <= 3 * 168, "register split exceeds the launch budget");
constexpr int kAllocWarp = 8;   // TMEM allocation / release
constexpr int kTmaWarp = 9;     // scheduler + TMA producer
constexpr int kIssueWarp = 10;  // MMA issue (one thread)

// barrier indices
enum : int {
  B_Q_FULL = 0, B_Q_EMPTY = 2, B_S_FULL = 4, B_O_FULL = 6, B_SCHED_FULL = 8, B_SCHED_EMPTY = 10,
  B_FINAL = 12, B_P_DONE = 14, B_O_READ = 16, B_STALL = 18,
  B_KV = 20  // then kStages "full" and kStages "empty" barriers
};

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;               // 128-byte swizzle atoms along d
  static constexpr int kTileBytes = BN * D * 2;        // a K or V tile; also a Q sub-tile (BM == BN)
  static constexpr int kStages = D == 128 ? 5 : 10;    // K/V ring depth (fills 224 KB with Q)
  // one barrier for V_j and K_{j+1} (one wait and one release per tile instead of
  // two): 5 % faster at d = 64, 0.3 % slower at d = 128 (measured A/B), so d = 64 only
  static constexpr bool kGroupKV = D == 64;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  static constexpr int kNumBars = B_KV + 2 * kStages;
  static constexpr int kOffInfo = kOffBar + kNumBars * 8;
  static constexpr int kOffMisc = kOffInfo + 2 * 96;   // two UnitInfo slots
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kColS = 0;
  static constexpr int kColO = 256;
  static_assert(kColO + 2 * D <= 512, "TMEM columns");
};

struct UnitInfo {
  uint32_t w;            // work id; >= num_tiles: no more work
  int32_t b, row0, h, g;
  int32_t len_k, off_q, off_k, off_v, off_o, off_s, shift, lo_shift;
  int32_t n_kv[2];       // KV tiles each sub-tile visits in this entry
  int32_t t_lo[2];       // loop index of each sub-tile's first tile (when n_kv > 0)
  int32_t n_rows[2];     // valid query rows of each sub-tile
  int32_t kv_lo;         // absolute KV tile of loop index 0
  int32_t n_tiles;       // KV tiles loaded for this entry
  int32_t part_slot;     // partial-result slot, -1 for a whole pair
  int32_t pad[2];
};
static_assert(sizeof(UnitInfo) == 96, "UnitInfo is 96 bytes");


__device__ __forceinline__ UnitInfo make_unit(const FwdParams& p, uint32_t w, uint32_t num_tiles) {
  UnitInfo u;
  u.w = w;
  u.b = u.row0 = u.h = u.g = 0;
  u.len_k = u.off_q = u.off_k = u.off_v = u.off_o = u.off_s = u.shift = u.lo_shift = 0;
  u.n_kv[0] = u.n_kv[1] = u.t_lo[0] = u.t_lo[1] = u.n_rows[0] = u.n_rows[1] = 0;
  u.kv_lo = u.n_tiles = 0;
  u.part_slot = -1;
  u.pad[0] = u.pad[1] = 0;
  if (w >= num_tiles) return u;
  int pair_idx, head;
  work_to_unit(p.header, w, p.h_q, p.h_kv, pair_idx, head);
  const PairRec pr = p.pairs[pair_idx];
  const SeqMeta m = p.meta[pr.b];
  u.b = pr.b;
  u.row0 = pr.row0;
  u.h = head;
  u.g = u.h / (p.h_q / p.h_kv);
  u.len_k = m.len_k;
  u.off_q = m.off_q; u.off_k = m.off_k; u.off_v = m.off_v; u.off_o = m.off_o; u.off_s = m.off_s;
  u.shift = m.shift;
  u.lo_shift = m.lo_shift;
  // absolute KV tile range [first, end) of each sub-tile: from the tile holding
  // its first row's lowest visible key to the one holding its last row's highest
  int first[2], end[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r_begin = pr.row0 + t * BM;
    const int rows = max(0, min(BM, m.len_q - r_begin));
    u.n_rows[t] = rows;
    first[t] = (int)(max64(0, (int64_t)r_begin + m.lo_shift) / BN);
    end[t] = 0;
    if (rows > 0) {
      const int64_t kmax = min64((int64_t)m.len_k, (int64_t)(r_begin + rows - 1) + m.shift + 1);
      end[t] = kmax > 0 ? (int)((kmax + BN - 1) / BN) : 0;
    }
  }
  // the pair spans n tiles [first[0], max end); part i of a pair split into `parts`
  // covers [i n / parts, (i + 1) n / parts) of that span
  const int f_pair = first[0];
  const int n_pair = max(0, max(end[0], end[1]) - f_pair);
  const int parts = pr.split & 0xff, part = pr.split >> 8;
  int lo = f_pair, hi = f_pair + n_pair;
  if (parts > 1) {
    lo = f_pair + (int)(((int64_t)part * n_pair) / parts);
    hi = f_pair + (int)(((int64_t)(part + 1) * n_pair) / parts);
    u.part_slot = pr.part;
  }
  int start[2], kv_lo = hi;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    start[t] = max(lo, first[t]);
    u.n_kv[t] = max(0, min(hi, end[t]) - start[t]);
    if (u.n_kv[t] > 0) kv_lo = min(kv_lo, start[t]);
  }
  u.kv_lo = kv_lo;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    u.t_lo[t] = u.n_kv[t] > 0 ? start[t] - kv_lo : 0;
    if (u.n_kv[t] > 0) u.n_tiles = max(u.n_tiles, u.t_lo[t] + u.n_kv[t]);
  }
  return u;
}

// WIN: some sequence may carry a left window, so a sub-tile's KV range may start
// after the unit's first tile (compiled out otherwise; the window-free variant keeps
// the shorter issue loop and mask)
template <int D, bool BF16, bool WIN>
__global__ void __launch_bounds__(kThreadsTC, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + C::kOffInfo);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);
  const Sync sy{sbase + (uint32_t)C::kOffBar, abort_flag, p.status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(sy.bar(B_Q_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_Q_EMPTY + t), 1);
      ptx::mbar_init(sy.bar(B_S_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_O_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_SCHED_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_SCHED_EMPTY + t), 9);  // 8 softmax warps + the issuing thread
      ptx::mbar_init(sy.bar(B_FINAL + t), 1);
      ptx::mbar_init(sy.bar(B_P_DONE + t), 4);   // one arrival per warp of the sub-tile
      ptx::mbar_init(sy.bar(B_STALL + t), 1);    // never arrived on (test hook)
      ptx::mbar_init(sy.bar(B_O_READ + t), 4);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(sy.bar(B_KV + s), 1);
      ptx::mbar_init(sy.bar(B_KV + C::kStages + s), 1);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  if (warp == kAllocWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t num_tiles = p.header[kHdrNumTiles];
  if (threadIdx.x == 0) THD_CTA_STAMP(0);

  if (warp >= 8) {
    ptx::setmaxnreg_dec<kRegsControl>();
    if (warp == kTmaWarp && lane == 0) {
      // ---------------------------------------------- scheduler + TMA producer
      uint32_t q_uses[2] = {0, 0};
      uint32_t kv_it = 0;
      // per ring slot: ever filled; its last fill released by the empty barrier of the
      // next slot (else its own); parity of that release phase. Per barrier slot:
      // parity of the empty phases handed out and of the full phases armed; armed once
      uint32_t filled = 0, rel_next = 0, rel_par = 0, e_cnt = 0, f_cnt = 0, f_used = 0;
      for (uint32_t it = 0;; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_EMPTY + slot, ((it >> 1) & 1u) ^ 1u)) break;
        const uint32_t w = atomicAdd(p.counter, 1u);
        const UnitInfo u = make_unit(p, w, num_tiles);
        THD_UNIT_STAMP(it, 0);
        THD_UNIT_INFO(it, ((unsigned long long)w << 32) | (uint32_t)u.n_tiles);
        info[slot] = u;
        ptx::mbar_arrive(sy.bar(B_SCHED_FULL + slot));
        if (w >= num_tiles) break;
        bool ok = true;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || u.n_kv[t] == 0) continue;
          if (!(ok = sy.wait(B_Q_EMPTY + t, (q_uses[t] & 1u) ^ 1u))) break;
          ++q_uses[t];
          const uint32_t qbar = sy.bar(B_Q_FULL + t);
          ptx::mbar_arrive_expect_tx(qbar, C::kTileBytes);
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            ptx::tma_load_3d(sbase + C::kOffQ + t * C::kTileBytes + hf * BM * 128, &tm_q, qbar, hf * 64, u.h,
                             u.off_q + u.row0 + t * BM);
        }
        const int n_tiles = u.n_tiles;
        if constexpr (!C::kGroupKV) {
          // one full and one empty barrier per ring slot, K_j then V_j
          for (int j = 0; j < n_tiles && ok; ++j) {
#pragma unroll
            for (int kv = 0; kv < 2; ++kv) {
              const int stage = (int)(kv_it % C::kStages);
              if (!(ok = sy.wait(B_KV + C::kStages + stage, ((kv_it / C::kStages) & 1u) ^ 1u))) break;
              ++kv_it;
              const uint32_t fbar = sy.bar(B_KV + stage);
              ptx::mbar_arrive_expect_tx(fbar, C::kTileBytes);
              const void* map = kv == 0 ? static_cast<const void*>(&tm_k) : static_cast<const void*>(&tm_v);
              const int row = (kv == 0 ? u.off_k : u.off_v) + (u.kv_lo + j) * BN;
#pragma unroll
              for (int hf = 0; hf < C::kHalves; ++hf)
                ptx::tma_load_3d(sbase + C::kOffKV + stage * C::kTileBytes + hf * BN * 128, map, fbar, hf * 64,
                                 u.g, row);
            }
          }
        } else {
          // fills i = 0 .. 2n-1 in order K_0, V_0, K_1, ..., V_{n-1} (K_j = 2j, V_j = 2j+1).
          // A group of fills shares the full and the empty barrier of its last fill's
          // slot: the groups are {K_0}, {V_0, K_1}, ..., {V_{n-1}}, as the issuing
          // thread consumes them
          for (int i0 = 0; i0 < 2 * n_tiles && ok;) {
            const uint32_t nf = ((i0 & 1) && i0 + 1 < 2 * n_tiles) ? 2u : 1u;
            const int gs = (int)((kv_it + nf - 1) % C::kStages);
            for (uint32_t q = 0; q < nf && ok; ++q) {
              const int x = (int)((kv_it + q) % C::kStages);
              if ((filled >> x) & 1u)
                ok = sy.wait(B_KV + C::kStages + (((rel_next >> x) & 1u) ? (x + 1) % C::kStages : x),
                             (rel_par >> x) & 1u);
            }
            if (!ok) break;
            const uint32_t ep = (e_cnt >> gs) & 1u;   // parity of the empty phase that releases this group
            e_cnt ^= 1u << gs;
            const uint32_t fbar = sy.bar(B_KV + gs);
            ptx::mbar_arrive_expect_tx(fbar, nf * (uint32_t)C::kTileBytes);
            f_cnt ^= 1u << gs;
            f_used |= 1u << gs;
            for (uint32_t q = 0; q < nf; ++q) {
              const int x = (int)((kv_it + q) % C::kStages);
              const int i = i0 + (int)q;
              filled |= 1u << x;
              rel_next = (rel_next & ~(1u << x)) | ((x != gs ? 1u : 0u) << x);
              rel_par = (rel_par & ~(1u << x)) | (ep << x);
              const bool is_v = i & 1;
              const void* map = is_v ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
              const int row = (is_v ? u.off_v : u.off_k) + (u.kv_lo + (i >> 1)) * BN;
  #pragma unroll
              for (int hf = 0; hf < C::kHalves; ++hf)
                ptx::tma_load_3d(sbase + C::kOffKV + x * C::kTileBytes + hf * BN * 128, map, fbar, hf * 64, u.g, row);
            }
            kv_it += nf;
            i0 += (int)nf;
          }
        }
        THD_UNIT_STAMP(it, 1);
        if (!ok) break;
      }
      // loads complete whether or not anyone consumes them; on an abort wait for
      // the ones still in flight before the CTA may exit
      if (*abort_flag) {
        for (int s = 0; s < C::kStages; ++s) {
          // the last phase armed on full barrier s
          bool armed;
          uint32_t parity;
          if constexpr (C::kGroupKV) {
            armed = (f_used >> s) & 1u;
            parity = ((f_cnt >> s) & 1u) ^ 1u;
          } else {
            armed = kv_it > (uint32_t)s;
            const uint32_t last = armed ? (kv_it - 1 - (uint32_t)s) / C::kStages * C::kStages + (uint32_t)s : 0u;
            parity = (last / C::kStages) & 1u;
          }
          if (armed) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(sy.bar(B_KV + s), parity) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
        for (int t = 0; t < 2; ++t) {
          if (q_uses[t] == 0) continue;
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(sy.bar(B_Q_FULL + t), (q_uses[t] - 1) & 1u) &&
                 ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    if (warp == kIssueWarp && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      // One thread issues for both sub-tiles, in the order
      //   QK0(0), QK1(0) | PV0(0), QK0(1), PV1(0), QK1(1) | PV0(1), QK0(2), ...
      // so the two sub-tiles' batches B_t(j) = {PV_t(j), QK_t(j+1)} alternate on
      // the tensor core and each softmax runs while the other sub-tile's MMAs
      // execute. Everything a batch needs except P (V_j, K_{j+1}) is waited for
      // first, then P_t(j), then the batch is issued back to back. The commit that
      // signals S_t(j+1) also covers PV_t(j), and P_t(j) (which overwrites S_t) is
      // read before QK_t(j+1) rewrites S_t because both are issued by this thread
      // in that order.
      constexpr uint32_t kIdescQK = ptx::idesc_f16(BF16, BM, BN, false);
      constexpr uint32_t kIdescPV = ptx::idesc_f16(BF16, BM, D, true);
      // descriptors of the operand bases; the start-address field (bits 0-13,
      // address >> 4) of each instruction's operand is the base plus a small offset
      // that stays inside the field, so a 64-bit add of (offset >> 4) selects it
      const uint64_t dq0 = ptx::sdesc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t dkv0 = ptx::sdesc_sw128(sbase + C::kOffKV, 16, 1024);
      const uint64_t dv0 = ptx::sdesc_sw128(sbase + C::kOffKV, BN * 128, 1024);
      auto issue_qk = [&](int t, int kstage) {
        const uint64_t qa = dq0 + (uint64_t)((t * C::kTileBytes) >> 4);
        const uint64_t ka = dkv0 + (uint64_t)((kstage * C::kTileBytes) >> 4);
        const uint32_t dS = tmem + (uint32_t)(C::kColS + t * BN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * BN * 128 + (kk & 3) * 32) >> 4);
          ptx::mma_ss(dS, qa + off, ka + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V over the first 16*nk keys: P from TMEM (8 columns per 16
      // keys), V MN-major (d contiguous): 8-key groups 1024 B apart, 64-wide d atoms
      // BN*128 B apart
      auto issue_pv = [&](int t, int vstage, bool accumulate, int nk) {
        const uint64_t va = dv0 + (uint64_t)((vstage * C::kTileBytes) >> 4);
        const uint32_t dO = tmem + (uint32_t)(C::kColO + t * D);
        const uint32_t aP = tmem + (uint32_t)(C::kColS + t * BN);
        if (nk == BN / 16) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            ptx::mma_ts(dO, aP + kk * 8, va + (uint64_t)(kk * 128), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        } else {
          for (int kk = 0; kk < nk; ++kk)
            ptx::mma_ts(dO, aP + kk * 8, va + (uint64_t)(kk * 128), kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      // ring slot and phase of a fill (one barrier pair per slot); with kGroupKV a
      // group of fills ({K_0}, {V_j, K_{j+1}}, {V_{n-1}}) is signalled and released by
      // the barriers of its last fill's slot, whose full phases are counted per slot
      // (parity bit in f_par)
      auto kv_stage = [](uint32_t fill) { return (int)(fill % C::kStages); };
      auto kv_phase = [](uint32_t fill) { return (fill / C::kStages) & 1u; };
      uint32_t f_par = 0;
      auto wait_group = [&](int gs) -> bool {
        const bool r = sy.wait(B_KV + gs, (f_par >> gs) & 1u);
        f_par ^= 1u << gs;
        return r;
      };
      uint32_t q_uses[2] = {0, 0}, p_waits[2] = {0, 0}, o_reads_seen[2] = {0, 0}, o_read_waits[2] = {0, 0};
      uint32_t kv_base = 0;
      bool issued_any = false, ok = true;
      // first QK of sub-tile t (its S_t(start)) on the K tile in `kstage`
      auto first_qk = [&](int t, int kstage, int n) -> bool {
        if (!sy.wait(B_Q_FULL + t, (q_uses[t]++) & 1u)) return false;
        ptx::tc_fence_after();
        issue_qk(t, kstage);
        ptx::tc_commit(sy.bar(B_S_FULL + t));
        if (n == 1) ptx::tc_commit(sy.bar(B_Q_EMPTY + t));
        return true;
      };
      // test hook: a wait nothing completes, bounded at 100 ms, exercises the abort path
      if (p.test_stall) ok = sy.wait(B_STALL, 0, 100000000ull);
      for (uint32_t it = 0; ok; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
        const UnitInfo u = info[slot];
        ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
        if (u.w >= num_tiles) break;
        THD_UNIT_STAMP(it, 2);
        // sub-tile t visits loop indices [tl[t], te[t]); with a left window the
        // second sub-tile may start later than the first
        const int nt[2] = {u.n_kv[0], u.n_kv[1]};
        const int tl[2] = {WIN ? u.t_lo[0] : 0, WIN ? u.t_lo[1] : 0};
        const int te[2] = {tl[0] + nt[0], tl[1] + nt[1]};
        const int n_tiles = u.n_tiles;
        if (n_tiles == 0) continue;
        if constexpr (C::kGroupKV) ok = wait_group(kv_stage(kv_base));
        else ok = sy.wait(B_KV + kv_stage(kv_base), kv_phase(kv_base));
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (ok && nt[t] > 0 && (!WIN || tl[t] == 0)) ok = first_qk(t, kv_stage(kv_base), nt[t]);
        if (!ok) break;
        ptx::tc_commit(sy.bar(B_KV + C::kStages + kv_stage(kv_base)));
        issued_any = true;
        THD_UNIT_STAMP(it, 3);
        for (int j = 0; j < n_tiles && ok; ++j) {
          THD_TRACE_STAMP(2, j, 0, it);
          const uint32_t vfill = kv_base + 2u * (uint32_t)j + 1u;
          const uint32_t kfill = kv_base + 2u * (uint32_t)(j + 1);
          const int vstage = kv_stage(vfill);
          const int kstage = kv_stage(kfill);
          const bool kmore = j + 1 < n_tiles;
          const int gstage = kmore ? kstage : vstage;
          if constexpr (C::kGroupKV) ok = wait_group(gstage);
          else ok = sy.wait(B_KV + vstage, kv_phase(vfill)) && (!kmore || sy.wait(B_KV + kstage, kv_phase(kfill)));
          if (!ok) break;
          THD_TRACE_STAMP(2, j, 1, it);
          // keys of this tile that exist: PV runs over ceil(valid/16) steps of 16
          // keys, and the at most 15 rows between valid and that bound are zeroed
          // (pad rows may hold NaN and 0 * NaN = NaN); whole 128-byte rows, so
          // swizzle-agnostic
          int nk = BN / 16;
          const int jj = u.kv_lo + j;            // absolute KV tile
          if ((jj + 1) * BN > u.len_k) {
            const int valid = u.len_k - jj * BN;
            nk = (valid + 15) >> 4;
            const int zrows = nk * 16 - valid;
            if (zrows > 0) {
              uint8_t* vt = smem + C::kOffKV + vstage * C::kTileBytes;
              for (int hf = 0; hf < C::kHalves; ++hf)
                for (int idx = 0; idx < zrows * 8; ++idx)
                  *reinterpret_cast<uint4*>(vt + hf * BN * 128 + valid * 128 + idx * 16) = make_uint4(0, 0, 0, 0);
              ptx::fence_proxy_async_smem();
            }
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok || j < tl[t] || j >= te[t]) continue;
            // the previous unit's epilogue has read O_t before the first PV_t overwrites it
            while (ok && j == tl[t] && o_read_waits[t] < o_reads_seen[t])
              ok = sy.wait(B_O_READ + t, (o_read_waits[t]++) & 1u);
            ok = ok && sy.wait(B_P_DONE + t, (p_waits[t]++) & 1u);
            if (!ok) break;
            THD_TRACE_STAMP(2, j, 2 + 2 * t, it);
            ptx::tc_fence_after();
            issue_pv(t, vstage, j > tl[t], nk);
            if (j + 1 < te[t]) {
              issue_qk(t, kstage);
              ptx::tc_commit(sy.bar(B_S_FULL + t));
              if (j + 2 == te[t]) ptx::tc_commit(sy.bar(B_Q_EMPTY + t));
            } else {
              ptx::tc_commit(sy.bar(B_O_FULL + t));
            }
            THD_TRACE_STAMP(2, j, 3 + 2 * t, it);
          }
          if constexpr (WIN) {
#pragma unroll
            for (int t = 0; t < 2; ++t)
              if (ok && kmore && nt[t] > 0 && tl[t] == j + 1) ok = first_qk(t, kstage, nt[t]);
          }
          if (!ok) break;
          if constexpr (C::kGroupKV) {
            ptx::tc_commit(sy.bar(B_KV + C::kStages + gstage));
          } else {
            ptx::tc_commit(sy.bar(B_KV + C::kStages + vstage));
            if (kmore) ptx::tc_commit(sy.bar(B_KV + C::kStages + kstage));
          }
          THD_TRACE_STAMP(2, j, 6, it);
        }
        THD_UNIT_STAMP(it, 4);
        kv_base += 2u * (uint32_t)n_tiles;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (nt[t] > 0) ++o_reads_seen[t];
      }
      // drain every MMA this thread issued before TMEM is released
      if (issued_any) {
        ptx::tc_commit(sy.bar(B_FINAL));
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(sy.bar(B_FINAL), 0) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    // softmax warps poll briefly before the sleep-hinted waits: long polling takes
    // issue slots from the MMA-issuing and TMA threads on the same sub-partitions
    const Sync sw{sy.bar0, sy.abort_flag, sy.status, 4};
    // ---------------------------------------------------------- softmax, per sub-tile
    // Warpgroup t owns query rows [row0 + 128 t, row0 + 128 t + 128) of the unit:
    // its threads turn S_t into P_t in TMEM, rescale O_t when the running max
    // moves, and write O_t and the LSE at the end of the unit.
    const int t = warp >> 2;                    // sub-tile
    const int row = ((warp & 3) << 5) + lane;   // TMEM lane == query row within the sub-tile
    const uint32_t lane_bits = (uint32_t)((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_bits + (uint32_t)(C::kColS + t * BN);
    const uint32_t tO = tmem + lane_bits + (uint32_t)(C::kColO + t * D);
    const float sl2 = p.scale_log2;
    T* __restrict__ O = static_cast<T*>(p.o);
    // warp-level arrival on a barrier the issuing thread waits on (bounded), after
    // this thread's tcgen05 stores/loads are complete
    auto warp_arrive = [&](int b) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(b));
    };
    uint32_t s_cnt = 0, o_cnt = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = (int)(it & 1u);
      if (!sw.wait_warp(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
      // the slot stays claimed until the epilogue, which reads its fields again
      // instead of keeping them in registers through the tile loop
      const UnitInfo u = info[slot];
      if (u.w >= num_tiles) break;
      const int n = t ? u.n_kv[1] : u.n_kv[0];
      const int nrows = t ? u.n_rows[1] : u.n_rows[0];
      if (nrows == 0) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
        continue;
      }
      const int r = u.row0 + t * BM + row;      // row inside the sequence
      const bool live = row < nrows;
      const int kmax_row = (int)max64(0, min64((int64_t)u.len_k, (int64_t)r + u.shift + 1));
      const int kmin_row = WIN ? (int)max64(0, min64((int64_t)u.len_k, (int64_t)r + u.lo_shift)) : 0;
      const int jt0 = u.kv_lo + (WIN ? (t ? u.t_lo[1] : u.t_lo[0]) : 0);   // absolute tile of j = 0
      float m = -INFINITY, l = 0.f;
      bool ok = true;
#ifdef THD_FWD_TRACE
      const bool tr = (warp & 3) == 0 && lane == 0;
#define THD_SOFTMAX_STAMP(ev) do { if (tr) THD_TRACE_STAMP(t, j, ev, it); } while (0)
#else
#define THD_SOFTMAX_STAMP(ev) ((void)0)
#endif
      for (int j = 0; j < n; ++j) {
        THD_SOFTMAX_STAMP(0);
        if (!(ok = sw.wait_warp(B_S_FULL + t, (s_cnt++) & 1u))) break;
        ptx::tc_fence_after();
        THD_SOFTMAX_STAMP(1);
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, s[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_wait_ld(s[c]);
        THD_SOFTMAX_STAMP(2);
        const int lim = kmax_row - (jt0 + j) * BN;      // columns >= lim are not visible
        if (lim < BN) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= lim) s[c][i] = __float_as_uint(-INFINITY);
        }
        const int lim_lo = kmin_row - (jt0 + j) * BN;   // nor columns < lim_lo (left window)
        if (WIN && lim_lo > 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i < lim_lo) s[c][i] = __float_as_uint(-INFINITY);
        }
        // P against the running reference max m (base 2, scaled). Fast path: no
        // row max at all; it is valid while every p stays <= 2^15 (fp16-safe), which
        // holds if the row sum does (p >= 0). Slow path (the row's first visible
        // tile, or a sum above 2^15, or a non-finite sum): take the tile max, move
        // m if it rose by more than 8, rescale l and O, and recompute P.
        auto compute_p = [&](float mref, float& rs_out) {
          const uint64_t scale2 = ptx::f2_pack(sl2, sl2);
          const uint64_t shift2 = ptx::f2_pack(-mref, -mref);
          uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int hp = 0; hp < 2; ++hp) {       // keys [64*hp, 64*hp+64) -> P columns [32*hp, 32*hp+32)
            uint32_t pk[32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const int c = 2 * hp + c2;
                float x0, x1;
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])),
                                           scale2, shift2),
                               x0, x1);
                const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                sum2[(i >> 1) & 3] = ptx::f2_add(sum2[(i >> 1) & 3], ptx::f2_pack(p0, p1));
                pk[c2 * 16 + (i >> 1)] = pack2<BF16>(p0, p1);
              }
            ptx::tmem_st32(tS + 32 * hp, pk);
          }
          float a0, a1, b0, b1;
          ptx::f2_unpack(ptx::f2_add(sum2[0], sum2[1]), a0, a1);
          ptx::f2_unpack(ptx::f2_add(sum2[2], sum2[3]), b0, b1);
          rs_out = (a0 + a1) + (b0 + b1);
        };
        float rs = 0.f;
        bool slow = __any_sync(0xffffffffu, m == -INFINITY);
        if (!slow) {
          compute_p(m, rs);
          slow = __any_sync(0xffffffffu, !(rs <= 32768.f));
        }
        float alpha = 1.f;
        bool resc = false;
        if (slow) {
          // row max: 8 independent chains of 3-input max
          float acc[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaxf(__uint_as_float(s[0][q]), __uint_as_float(s[0][q + 8]));
#pragma unroll
          for (int i = 16; i < 128; i += 16)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              acc[q] = ptx::fmax3(acc[q], __uint_as_float(s[(i + q) >> 5][(i + q) & 31]),
                                  __uint_as_float(s[(i + q + 8) >> 5][(i + q + 8) & 31]));
          const float mx = ptx::fmax3(ptx::fmax3(acc[0], acc[1], acc[2]), ptx::fmax3(acc[3], acc[4], acc[5]),
                                      fmaxf(acc[6], acc[7]));
          // the reference max moves only when the tile max exceeds it by more than
          // 8, so O is rescaled rarely and p stays below 2^8 right after a move
          const float mt = mx * sl2;
          resc = mt > m + 8.0f;
          if (resc) {
            alpha = ptx::ex2(m - mt);
            m = mt;
          }
          compute_p(m == -INFINITY ? 0.f : m, rs);
        }
        l = l * alpha + rs;
        THD_SOFTMAX_STAMP(3);
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O_t already holds PV of tiles < j (the commit of S_t(j) covered PV_t(j-1))
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + 32 * c, o);
            ptx::tmem_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st32(tO + 32 * c, o);
          }
        }
        ptx::tmem_wait_st();
        THD_SOFTMAX_STAMP(4);
        warp_arrive(B_P_DONE + t);               // this warp's rows of P_t(j) (and O_t rescale) stored
        THD_SOFTMAX_STAMP(5);
      }
#undef THD_SOFTMAX_STAMP
      if (!ok) break;
      // epilogue: O = O_acc / l on live rows, LSE = (m + log2 l) * ln 2; dead rows 0 / -inf.
      // For half of a split pair the normalised partial O (fp32) and its base-2 LSE
      // go to the partial buffers instead; the combine kernel merges the halves.
      const volatile UnitInfo* ui = info + slot;
      const int e_part = ui->part_slot, e_off_o = ui->off_o, e_h = ui->h, e_off_s = ui->off_s;
      const int er = ui->row0 + t * BM + row;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
      const bool partial = e_part >= 0;
      const int urow = t * BM + row;            // row within the unit
      T* orow = O + (int64_t)(e_off_o + er) * p.stride_tok[3] + (int64_t)e_h * p.stride_head[3];
      float* prow = p.part_o + (((int64_t)e_part * p.h_q + e_h) * p.rows_per_unit + urow) * D;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (n > 0) {
        if (!sw.wait_warp(B_O_FULL + t, (o_cnt++) & 1u)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + 32 * c, o);
          ptx::tmem_wait_ld(o);
          if (live && partial) {
            float4* dst = reinterpret_cast<float4*>(prow + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                    __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
          } else if (live) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
        }
        // every thread's reads of O_t complete before the issuing thread's next PV_t
        warp_arrive(B_O_READ + t);
      } else if (live && partial) {
        float4* dst = reinterpret_cast<float4*>(prow);
#pragma unroll
        for (int q4 = 0; q4 < D / 4; ++q4) dst[q4] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else if (live) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int q4 = 0; q4 < D / 8; ++q4) dst[q4] = make_uint4(0, 0, 0, 0);
      }
      if (live && partial) {
        p.part_lse[((int64_t)e_part * p.h_q + e_h) * p.rows_per_unit + urow] =
            l > 0.f ? m + ptx::lg2(l) : -INFINITY;
      } else if (live) {
        const float lse = l > 0.f ? (m + ptx::lg2(l)) * 0.69314718055994530942f : -INFINITY;
        p.stats[(int64_t)(e_off_s + er) * p.stats_tok + (int64_t)e_h * p.stats_head] = lse;
      }
#ifdef THD_FWD_TRACE
      if ((warp & 3) == 0 && lane == 0) THD_UNIT_STAMP(it, 5 + t);
#endif
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) THD_CTA_STAMP(1);
  if (warp == kAllocWarp) {
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}


template <int D, bool BF16, bool WIN>
cudaError_t launch_impl(const FwdParams& p, const thd_attn_desc_t& desc, int max_pairs, int num_sms,
                        cudaStream_t stream) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv;
  if (!encode_view(&tq, p.q, BF16, D, desc.h_q, desc.cap_rows[0], desc.stride_head[0], desc.stride_tok[0]) ||
      !encode_view(&tk, p.k, BF16, D, desc.h_kv, desc.cap_rows[1], desc.stride_head[1], desc.stride_tok[1]) ||
      !encode_view(&tv, p.v, BF16, D, desc.h_kv, desc.cap_rows[2], desc.stride_head[2], desc.stride_tok[2]))
    return cudaErrorNotSupported;
  const int smem = C::kSmemBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, BF16, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = tc_grid_size(num_sms, max_pairs, desc.h_q);
  fwd_tc_kernel<D, BF16, WIN><<<grid, kThreadsTC, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_kernel_available() { return true; }

#ifdef THD_FWD_TRACE
// traced builds only: copy / clear the timeline of the last traced launch
extern "C" int thd_fwd_trace_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_fwd_trace, bytes < sizeof(g_fwd_trace) ? bytes : sizeof(g_fwd_trace));
}
extern "C" int thd_fwd_trace_clear() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fwd_trace) != cudaSuccess || cudaMemset(p, 0, sizeof(g_fwd_trace)) != cudaSuccess)
    return 1;
  if (cudaGetSymbolAddress(&p, g_fwd_units) != cudaSuccess || cudaMemset(p, 0, sizeof(g_fwd_units)) != cudaSuccess)
    return 1;
  if (cudaGetSymbolAddress(&p, g_fwd_cta) != cudaSuccess) return 1;
  return (int)cudaMemset(p, 0, sizeof(g_fwd_cta));
}
// unit timeline (g_fwd_units) followed by the CTA spans (g_fwd_cta)
extern "C" int thd_fwd_trace_units_read(void* host, size_t bytes) {
  if (bytes < sizeof(g_fwd_units) + sizeof(g_fwd_cta)) return 1;
  if (cudaMemcpyFromSymbol(host, g_fwd_units, sizeof(g_fwd_units)) != cudaSuccess) return 1;
  return (int)cudaMemcpyFromSymbol(static_cast<char*>(host) + sizeof(g_fwd_units), g_fwd_cta, sizeof(g_fwd_cta));
}
#endif
int tc_grid_size(int num_sms, int max_pairs, int h_q) {
  // entries: at most two per pair (KV split)
  return (int)max64(1, min64((int64_t)num_sms, 2 * (int64_t)max_pairs * h_q));
}
int tc_rows_per_unit() { return 2 * BM; }
int tc_keys_per_tile() { return BN; }

cudaError_t launch_fwd_tc(const FwdParams& p, const thd_attn_desc_t& desc, int max_pairs, int num_sms,
                          cudaStream_t stream) {
  const bool bf16 = desc.dtype == THD_BF16;
  const bool win = p.has_window != 0;
#define THD_TC_LAUNCH(D_, B_)                                                     \
  return win ? launch_impl<D_, B_, true>(p, desc, max_pairs, num_sms, stream)     \
             : launch_impl<D_, B_, false>(p, desc, max_pairs, num_sms, stream)
  if (desc.d == 128) {
    if (bf16) THD_TC_LAUNCH(128, true);
    THD_TC_LAUNCH(128, false);
  }
  if (desc.d == 64) {
    if (bf16) THD_TC_LAUNCH(64, true);
    THD_TC_LAUNCH(64, false);
  }
#undef THD_TC_LAUNCH
  return cudaErrorNotSupported;
}

}  // namespace thd
