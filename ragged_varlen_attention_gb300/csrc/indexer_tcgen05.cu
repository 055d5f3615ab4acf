// Indexer scores on the tensor cores (sm_103a), the dense part of the indexer
// top-k: I_ij = sum_h w_ih * max(0, <q_ih, k_j>) for every visible (row, key)
// pair (Megatron-LM PR #14 "fix(dsa): align packed-CP indexer causal masks": the
// causal policy and q_causal_offset of the packed context-parallel chunks).
//
// Unit = 256 keys of one sequence (key-axis schedule, longest first), two 128-key
// sub-tiles K_0, K_1 [128 keys x d] resident in shared memory; the query rows that
// see any of its keys stream through a ring in groups of R = 128 / H rows with all
// H heads, and each streamed group feeds two tcgen05.mma chains S^T_t = K_t Q'^T
// (M = 128 keys, N = 128 (row, head) pairs, K = d): the group tile (32 KB at
// d = 128) is the large operand, so serving 256 keys per load halves the L2 traffic
// per FLOP. The score warps own one key of each sub-tile (TMEM lane) and 64
// (row, head) columns, so the reduction over heads, sum_h w_ih max(0, s), stays
// inside the thread; a warp stores 32 consecutive keys of a row (128 bytes). Two
// TMEM buffers (256 columns each) let the MMAs of group s + 1 run while group s is
// reduced.
//
// TMA: Q' as a {64 d, H heads, R rows} box of the [rows, H, d] view (128-byte
// swizzle: the box lands as 128 rows of 128 bytes, row = r * H + h, the same
// layout as a [128 x 64] tile), W as an {H, R} float32 box, K as {64, 128}.
// Only visible pairs are stored (key j < len_k, row i < len_q, j <= i + shift);
// the top-k kernel reads row i's keys below its causal limit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tc_common.cuh"
#include "tc_launch.h"

namespace thd {

namespace {

using tc::kWaitLimitNs;
using tc::Sync;

constexpr int kThreadsIx = 384;
constexpr int kAllocWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kIssueWarp = 10;

enum : int {
  B_IN_FULL = 0, B_IN_EMPTY = 1, B_S_FULL = 2, B_S_FREE = 4, B_SCHED_FULL = 6, B_SCHED_EMPTY = 8,
  B_FINAL = 10, B_RING = 11
};

template <int D, int H>
struct IxCfg {
  static constexpr int R = 128 / H;                 // query rows per group
  static constexpr int RW = 64 / H;                 // rows per score warpgroup
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;    // K tile, Q' tile
  static constexpr int kWBytes = R * H * 4;         // 512
  static constexpr int kStages = D == 128 ? 4 : 8;
  static constexpr int kOffK = 0;                   // K_0, K_1
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffW = kOffRing + kStages * kTileBytes;
  static constexpr int kOffBar = kOffW + kStages * kWBytes;
  static constexpr int kNumBars = B_RING + 2 * kStages;
  static constexpr int kOffInfo = kOffBar + kNumBars * 8;
  static constexpr int kOffMisc = kOffInfo + 2 * 48;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory");
  static_assert(R * H == 128 && RW * H == 64, "H must divide 64");
};

struct IxUnit {
  uint32_t w;
  int32_t b, k0, n_keys, len_q, len_k, shift, off_q, off_k, off_o, g0, n_steps;
};
static_assert(sizeof(IxUnit) == 48, "IxUnit is 48 bytes");

template <int R>
__device__ __forceinline__ IxUnit make_unit_ix(const IndexerParams& p, uint32_t w, uint32_t num_tiles) {
  IxUnit u;
  u.w = w;
  u.b = u.k0 = u.n_keys = u.len_q = u.len_k = u.shift = u.off_q = u.off_k = u.off_o = u.g0 = u.n_steps = 0;
  if (w >= num_tiles) return u;
  int pair, head;
  work_to_unit(p.header_k, w, 1, 1, pair, head);
  const PairRec pr = p.pairs_k[pair];
  const SeqMeta m = p.meta[pr.b];
  u.b = pr.b; u.k0 = pr.row0;
  u.n_keys = max(0, min(kIndexerKeysPerUnit, m.len_k - pr.row0));
  u.len_q = m.len_q; u.len_k = m.len_k; u.shift = m.shift;
  u.off_q = m.off_q; u.off_k = m.off_k; u.off_o = m.off_o;
  // rows that see a key of the tile: i >= k0 - shift
  const int64_t i_lo = max64(0, (int64_t)pr.row0 - m.shift);
  if (u.n_keys > 0 && i_lo < m.len_q) {
    u.g0 = (int)(i_lo / R);
    u.n_steps = (m.len_q + R - 1) / R - u.g0;
  }
  return u;
}

template <int D, int H>
__global__ void __launch_bounds__(kThreadsIx, 1)
    indexer_scores_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_w, const IndexerParams p, const uint32_t idesc) {
  using C = IxCfg<D, H>;
  constexpr int R = C::R, RW = C::RW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  IxUnit* info = reinterpret_cast<IxUnit*>(smem + C::kOffInfo);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 4);
  const Sync sy{sbase + (uint32_t)C::kOffBar, abort_flag, p.status};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t num_tiles = p.header_k[kHdrNumTiles];
  const uint32_t S = C::kStages;

  if (threadIdx.x == 0) {
    ptx::mbar_init(sy.bar(B_IN_FULL), 1);
    ptx::mbar_init(sy.bar(B_IN_EMPTY), 1);
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(sy.bar(B_S_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_S_FREE + t), 8);
      ptx::mbar_init(sy.bar(B_SCHED_FULL + t), 1);
      ptx::mbar_init(sy.bar(B_SCHED_EMPTY + t), 9);
    }
    ptx::mbar_init(sy.bar(B_FINAL), 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(sy.bar(B_RING + s), 1);
      ptx::mbar_init(sy.bar(B_RING + C::kStages + s), 8);   // released by the score warps
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_w);
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
    if (warp == kTmaWarp && lane == 0) {
      // ------------------------------------------------ scheduler + TMA producer
      uint32_t in_uses = 0, fill = 0;
      for (uint32_t it = 0;; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_EMPTY + slot, ((it >> 1) & 1u) ^ 1u)) break;
        const uint32_t w = atomicAdd(p.counter_k, 1u);
        const IxUnit u = make_unit_ix<R>(p, w, num_tiles);
        info[slot] = u;
        ptx::mbar_arrive(sy.bar(B_SCHED_FULL + slot));
        if (w >= num_tiles) break;
        if (u.n_steps == 0) continue;
        if (!sy.wait(B_IN_EMPTY, (in_uses & 1u) ^ 1u)) break;
        ++in_uses;
        ptx::mbar_arrive_expect_tx(sy.bar(B_IN_FULL), 2 * C::kTileBytes);
#pragma unroll
        for (int kt = 0; kt < 2; ++kt)
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            ptx::tma_load_2d(sbase + C::kOffK + kt * C::kTileBytes + hf * 128 * 128, &tm_k, sy.bar(B_IN_FULL),
                             hf * 64, u.off_k + u.k0 + kt * 128);
        bool ok = true;
        for (int s = 0; s < u.n_steps; ++s) {
          const int st = (int)(fill % S);
          if (!(ok = sy.wait(B_RING + C::kStages + st, ((fill / S) & 1u) ^ 1u))) break;
          ++fill;
          const uint32_t fb = sy.bar(B_RING + st);
          ptx::mbar_arrive_expect_tx(fb, C::kTileBytes + C::kWBytes);
          const int row = u.off_q + (u.g0 + s) * R;
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf)
            ptx::tma_load_3d(sbase + C::kOffRing + st * C::kTileBytes + hf * 128 * 128, &tm_q, fb, hf * 64, 0, row);
          ptx::tma_load_2d(sbase + C::kOffW + st * C::kWBytes, &tm_w, fb, 0, row);
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        for (uint32_t s = 0; s < S; ++s) {
          if (fill > s) {
            const uint32_t last = (fill - 1 - s) / S * S + s;
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(sy.bar(B_RING + (int)s), (last / S) & 1u) &&
                   ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
        if (in_uses > 0) {
          const uint64_t t0 = ptx::globaltimer_ns();
          while (!ptx::mbar_try_wait(sy.bar(B_IN_FULL), (in_uses - 1) & 1u) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    if (warp == kIssueWarp && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      const uint64_t dk = ptx::sdesc_sw128(sbase + C::kOffK, 16, 1024);
      const uint64_t dq = ptx::sdesc_sw128(sbase + C::kOffRing, 16, 1024);
      uint32_t in_uses = 0, fill = 0, uses[2] = {0, 0}, gstep = 0;
      bool issued_any = false, ok = true;
      for (uint32_t it = 0; ok; ++it) {
        const int slot = (int)(it & 1u);
        if (!sy.wait(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
        const IxUnit u = info[slot];
        ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
        if (u.w >= num_tiles) break;
        if (u.n_steps == 0) continue;
        if (!(ok = sy.wait(B_IN_FULL, (in_uses++) & 1u))) break;
        for (int s = 0; s < u.n_steps && ok; ++s, ++fill, ++gstep) {
          const int st = (int)(fill % S);
          const int b = (int)(gstep & 1u);
          ok = sy.wait(B_RING + st, (fill / S) & 1u);
          if (ok && uses[b] > 0) ok = sy.wait(B_S_FREE + b, (uses[b] - 1) & 1u);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint64_t qa = dq + (uint64_t)((st * C::kTileBytes) >> 4);
#pragma unroll
          for (int kt = 0; kt < 2; ++kt) {
            const uint64_t ka = dk + (uint64_t)((kt * C::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = (uint64_t)((((kk >> 2) * 128 * 128) + (kk & 3) * 32) >> 4);
              ptx::mma_ss(tmem + (uint32_t)(b * 256 + kt * 128), ka + off, qa + off, idesc, kk > 0 ? 1u : 0u);
            }
          }
          ptx::tc_commit(sy.bar(B_S_FULL + b));
          ++uses[b];
          issued_any = true;
          if (s + 1 == u.n_steps) ptx::tc_commit(sy.bar(B_IN_EMPTY));
        }
      }
      if (issued_any) {
        ptx::tc_commit(sy.bar(B_FINAL));
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(sy.bar(B_FINAL), 0) && ptx::globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- score warps: key = TMEM lane
    const int wg = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_bits = (uint32_t)((warp & 3) << 5) << 16;
    uint32_t fill = 0, uses[2] = {0, 0}, gstep = 0;
    for (uint32_t it = 0;; ++it) {
      const int slot = (int)(it & 1u);
      if (!sy.wait_warp(B_SCHED_FULL + slot, (it >> 1) & 1u)) break;
      const IxUnit u = info[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sy.bar(B_SCHED_EMPTY + slot));
      if (u.w >= num_tiles) break;
      bool ok = true;
      for (int s = 0; s < u.n_steps; ++s, ++fill, ++gstep) {
        const int st = (int)(fill % S);
        const int b = (int)(gstep & 1u);
        ok = sy.wait_warp(B_S_FULL + b, (uses[b]++) & 1u) && sy.wait_warp(B_RING + st, (fill / S) & 1u);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t v[2][2][32];                       // [key sub-tile][column chunk]
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          const uint32_t ta = tmem + lane_bits + (uint32_t)(b * 256 + kt * 128 + wg * 64);
          ptx::tmem_ld32(ta, v[kt][0]);
          ptx::tmem_ld32(ta + 32, v[kt][1]);
        }
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          ptx::tmem_wait_ld(v[kt][0]);
          ptx::tmem_wait_ld(v[kt][1]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sy.bar(B_S_FREE + b));
        const float* wt = reinterpret_cast<const float*>(smem + C::kOffW + st * C::kWBytes);
        const int i0 = (u.g0 + s) * R + wg * RW;    // first query row of this warpgroup's columns
        float acc[2][RW];
#pragma unroll
        for (int rl = 0; rl < RW; ++rl) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int hh = 0; hh < H; ++hh) {
            const int c = rl * H + hh;
            const float wv = wt[(wg * RW + rl) * H + hh];
            a0 = fmaf(wv, fmaxf(__uint_as_float(v[0][c >> 5][c & 31]), 0.f), a0);
            a1 = fmaf(wv, fmaxf(__uint_as_float(v[1][c >> 5][c & 31]), 0.f), a1);
          }
          acc[0][rl] = a0;
          acc[1][rl] = a1;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sy.bar(B_RING + C::kStages + st));
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          const int jr = kt * 128 + row;               // key within the unit
          const int j = u.k0 + jr;
#pragma unroll
          for (int rl = 0; rl < RW; ++rl) {
            const int i = i0 + rl;
            if (jr < u.n_keys && i < u.len_q && (int64_t)j <= (int64_t)i + u.shift)
              p.scores[(int64_t)(u.off_o + i) * p.score_row + j] = acc[kt][rl];
          }
        }
      }
      if (!ok) break;
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

template <int D, int H>
cudaError_t launch_ix(const IndexerParams& p, const thd_indexer_desc_t& d, int max_pairs_k, int num_sms,
                      cudaStream_t stream) {
  using C = IxCfg<D, H>;
  const CUtensorMapDataType ty = d.dtype == THD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tw;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)d.cap_rows_q};
    const cuuint64_t str[2] = {(cuuint64_t)(d.stride_head_q * 2), (cuuint64_t)(d.stride_tok_q * 2)};
    const cuuint32_t box[3] = {64, (cuuint32_t)H, (cuuint32_t)C::R};
    if (!tc_host::encode_tiled(&tq, p.q, ty, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorNotSupported;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)d.cap_rows_k};
    const cuuint64_t str[1] = {(cuuint64_t)(d.stride_tok_k * 2)};
    const cuuint32_t box[2] = {64, 128};
    if (!tc_host::encode_tiled(&tk, p.k, ty, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorNotSupported;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)d.cap_rows_q};
    const cuuint64_t str[1] = {(cuuint64_t)(d.stride_tok_w * 4)};
    const cuuint32_t box[2] = {(cuuint32_t)H, (cuuint32_t)C::R};
    if (!tc_host::encode_tiled(&tw, p.w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorNotSupported;
  }
  const int smem = C::kSmemBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_tc_kernel<D, H>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const uint32_t idesc = d.dtype == THD_BF16 ? ptx::idesc_f16(true, 128, 128, false) : ptx::idesc_f16(false, 128, 128, false);
  const int grid = (int)max64(1, min64((int64_t)num_sms, (int64_t)max_pairs_k));
  indexer_scores_tc_kernel<D, H><<<grid, kThreadsIx, smem, stream>>>(tq, tk, tw, p, idesc);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_ix_h(const IndexerParams& p, const thd_indexer_desc_t& d, int max_pairs_k, int num_sms,
                        cudaStream_t stream) {
  switch (d.heads) {
    case 4: return launch_ix<D, 4>(p, d, max_pairs_k, num_sms, stream);
    case 8: return launch_ix<D, 8>(p, d, max_pairs_k, num_sms, stream);
    case 16: return launch_ix<D, 16>(p, d, max_pairs_k, num_sms, stream);
    case 32: return launch_ix<D, 32>(p, d, max_pairs_k, num_sms, stream);
    case 64: return launch_ix<D, 64>(p, d, max_pairs_k, num_sms, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

bool indexer_tc_applicable(const thd_indexer_desc_t& d) {
  if (d.dtype != THD_BF16 && d.dtype != THD_FP16) return false;
  if (d.d != 64 && d.d != 128) return false;
  if (d.heads != 4 && d.heads != 8 && d.heads != 16 && d.heads != 32 && d.heads != 64) return false;
  if (d.stride_tok_q <= 0 || d.stride_head_q <= 0 || d.stride_tok_k <= 0 || d.stride_tok_w <= 0) return false;
  if ((d.stride_tok_q * 2) % 16 || (d.stride_head_q * 2) % 16 || (d.stride_tok_k * 2) % 16 || (d.stride_tok_w * 4) % 16)
    return false;
  return true;
}

cudaError_t launch_indexer_scores_tc(const IndexerParams& p, const thd_indexer_desc_t& d, int max_pairs_k,
                                     int num_sms, cudaStream_t stream) {
  if (d.d == 128) return launch_ix_h<128>(p, d, max_pairs_k, num_sms, stream);
  if (d.d == 64) return launch_ix_h<64>(p, d, max_pairs_k, num_sms, stream);
  return cudaErrorNotSupported;
}

}  // namespace thd
