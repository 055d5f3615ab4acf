// Indexer top-k kernels: a SIMT score kernel (any H <= 128, d <= 128; fp32
// arithmetic) and the per-row top-k selection shared by every score path.
//
// Scores (lightning-indexer form, see thd_indexer_topk in thd_attn.h):
// I_ij = sum_h w_ih * max(0, <q_ih, k_j>) for the visible prefix j < kmax_i of
// each row (the attention forward's mask policy and q_causal_offset; Megatron-LM
// PR #14 "fix(dsa): align packed-CP indexer causal masks"). Each output row owns a
// float32 row of the workspace; key j's score sits at column j.
//
// Top-k (one CTA per row at a time, persistent over all rows of the scheduled units):
// scores are mapped to order-preserving unsigned keys, the k-th largest key is
// found by a three-pass radix select over 11 + 11 + 10 bits (shared-memory
// histograms), every key above that threshold and the lowest-numbered keys equal
// to it are gathered (exactly k), and the k entries are sorted by descending score
// then ascending key number with a bitonic sort in shared memory. Rows with at
// most k visible keys skip the select and sort all of them. Score rows are read
// as float4; the first histogram pass aggregates equal bins within a warp
// (scores share few high bits), and the gather takes every element above the
// threshold with one atomic slot each, switching to an ordered scan only when
// more scores equal the threshold than slots remain.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "convert.cuh"
#include "internal.h"

namespace thd {

namespace {

constexpr int kScoreThreads = 256;
constexpr int kTopkThreads = 256;

// ------------------------------------------------------------------- scores (SIMT)
template <typename T>
__global__ void __launch_bounds__(kScoreThreads) indexer_scores_simt_kernel(IndexerParams p) {
  extern __shared__ float qs[];              // [H][d] of the current row, then w [H]
  const int H = p.heads, d = p.d;
  float* ws = qs + H * d;
  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ K = static_cast<const T*>(p.k);
  const uint32_t items = p.header[kHdrNumTiles] * (uint32_t)kIndexerRowsPerUnit;
  for (uint32_t item = blockIdx.x; item < items; item += gridDim.x) {
    int pair, head;
    work_to_unit(p.header, item / kIndexerRowsPerUnit, 1, 1, pair, head);
    const PairRec pr = p.pairs[pair];
    const SeqMeta m = p.meta[pr.b];
    {
      const int rr = (int)(item % kIndexerRowsPerUnit);
      if (pr.row0 + rr >= m.len_q) continue;      // uniform across the block
      const int r = pr.row0 + rr;
      __syncthreads();
      for (int x = threadIdx.x; x < H * d; x += blockDim.x) {
        const int h = x / d, e = x % d;
        qs[x] = to_f32(Q[(int64_t)(m.off_q + r) * p.q_tok + (int64_t)h * p.q_head + e]);
      }
      for (int h = threadIdx.x; h < H; h += blockDim.x) ws[h] = p.w[(int64_t)(m.off_q + r) * p.w_tok + h];
      __syncthreads();
      const int kmax = (int)max64(0, min64((int64_t)m.len_k, (int64_t)r + m.shift + 1));
      float* srow = p.scores + (int64_t)(m.off_o + r) * p.score_row;
      for (int j = threadIdx.x; j < kmax; j += blockDim.x) {
        const T* krow = K + (int64_t)(m.off_k + j) * p.k_tok;
        float score = 0.f;
        for (int h0 = 0; h0 < H; h0 += 32) {
          float dot[32];
#pragma unroll
          for (int hh = 0; hh < 32; ++hh) dot[hh] = 0.f;
          for (int e0 = 0; e0 < d; e0 += 32) {
            float kr[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) kr[e] = e0 + e < d ? to_f32(krow[e0 + e]) : 0.f;
#pragma unroll
            for (int hh = 0; hh < 32; ++hh) {
              if (h0 + hh < H) {
                const float* qh = qs + (h0 + hh) * d + e0;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (e0 + e < d) dot[hh] = fmaf(qh[e], kr[e], dot[hh]);
              }
            }
          }
#pragma unroll
          for (int hh = 0; hh < 32; ++hh)
            if (h0 + hh < H) score = fmaf(ws[h0 + hh], fmaxf(dot[hh], 0.f), score);
        }
        srow[j] = score;
      }
    }
  }
}

// ------------------------------------------------------------------------ top-k
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;              // -0 ranks with +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// inclusive suffix sums of hist[0..n) (n a multiple of blockDim.x) into hist, so
// hist[b] = number of elements in bins >= b
__device__ void suffix_sums(uint32_t* hist, int n, uint32_t* scratch) {
  const int per = n / blockDim.x;
  const int t = threadIdx.x;
  // each thread owns bins [n - (t+1)*per, n - t*per): thread 0 the highest
  uint32_t local = 0;
  for (int x = 0; x < per; ++x) local += hist[n - t * per - 1 - x];
  scratch[t] = local;
  __syncthreads();
  // exclusive prefix over threads (thread order = descending bins), by one warp
  if (t < 32) {
    uint32_t carry = 0;
    for (int base = 0; base < (int)blockDim.x; base += 32) {
      uint32_t v = scratch[base + t];
      uint32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (t >= o) incl += y;
      }
      scratch[base + t] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  uint32_t run = scratch[t];
  for (int x = 0; x < per; ++x) {
    const int bin = n - t * per - 1 - x;
    run += hist[bin];
    hist[bin] = run;
  }
  __syncthreads();
}

// the bin b of hist (suffix sums) with hist[b] >= need > hist[b + 1]; need >= 1
__device__ __forceinline__ int find_bin(const uint32_t* hist, int n, uint32_t need, int* out) {
  for (int b = threadIdx.x; b < n; b += blockDim.x) {
    const uint32_t above = b + 1 < n ? hist[b + 1] : 0u;
    if (hist[b] >= need && above < need) *out = b;
  }
  __syncthreads();
  return *out;
}

__device__ __forceinline__ unsigned long long sort_key(uint32_t kk, int j) {
  return ((unsigned long long)(0xffffffffu - kk) << 32) | (uint32_t)j;
}

__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(IndexerParams p) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scratch[kTopkThreads];
  __shared__ unsigned long long sortbuf[kIndexerMaxTopk];
  __shared__ int sel_bin;
  __shared__ uint32_t n_gt, n_eq, eq_base;
  const uint32_t num_tiles = p.header[kHdrNumTiles];
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  const int topk = p.topk;
  const int stride4 = (int)blockDim.x * 4;
  // one row per CTA at a time: item = (scheduled unit, row within it)
  const uint32_t items = num_tiles * (uint32_t)kIndexerRowsPerUnit;
  for (uint32_t item = blockIdx.x; item < items; item += gridDim.x) {
    int pair, head;
    work_to_unit(p.header, item / kIndexerRowsPerUnit, 1, 1, pair, head);
    const PairRec pr = p.pairs[pair];
    const SeqMeta m = p.meta[pr.b];
    {
      const int rr = (int)(item % kIndexerRowsPerUnit);
      if (pr.row0 + rr >= m.len_q) continue;      // uniform across the CTA
      const int r = pr.row0 + rr;
      const int n = (int)max64(0, min64((int64_t)m.len_k, (int64_t)r + m.shift + 1));
      const float* srow = p.scores + (int64_t)(m.off_o + r) * p.score_row;   // 512-byte aligned
      const int n_out = min(n, topk);
      if (t == 0) { n_gt = 0; n_eq = 0; eq_base = 0; }
      __syncthreads();
      if (n <= topk) {
        for (int j = t; j < n; j += blockDim.x) sortbuf[j] = sort_key(order_key(srow[j]), j);
      } else {
        // radix select of the topk-th largest key over bits 31..21, 20..10, 9..0;
        // a warp walks 128 consecutive scores per step (float4 per lane), the loop
        // bound is warp-uniform so whole warps take part in the match below
        uint32_t prefix = 0, need = (uint32_t)topk, eq_total = 0;
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
          const int nb = 1 << widths[pass];
          for (int b = t; b < 2048; b += blockDim.x) hist[b] = 0;
          __syncthreads();
          const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (shifts[pass] + widths[pass]));
          for (int base = warp * 128; base < n; base += stride4) {
            const int j4 = base + lane * 4;
            const float4 v = *reinterpret_cast<const float4*>(srow + j4);
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t kk = order_key(vv[e]);
              const bool in = j4 + e < n && (kk & hi_mask) == prefix;
              const uint32_t bin = (kk >> shifts[pass]) & (uint32_t)(nb - 1);
              if (pass == 0) {
                // scores share few high bits: one atomic per distinct bin per warp
                const uint32_t key = in ? bin : 0xffffffffu;
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
              } else if (in) {
                atomicAdd(&hist[bin], 1u);
              }
            }
          }
          __syncthreads();
          suffix_sums(hist, nb, scratch);
          const int b = find_bin(hist, nb, need, &sel_bin);
          const uint32_t above = b + 1 < nb ? hist[b + 1] : 0u;
          eq_total = hist[b] - above;              // after the last pass: elements equal to the threshold
          need -= above;
          prefix |= (uint32_t)b << shifts[pass];
          __syncthreads();
        }
        const uint32_t thr = prefix;
        const uint32_t base_eq = (uint32_t)topk - need;
        // everything above the threshold; the equal ones too when all of them fit
        for (int base = warp * 128; base < n; base += stride4) {
          const int j4 = base + lane * 4;
          const float4 v = *reinterpret_cast<const float4*>(srow + j4);
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (j4 + e >= n) continue;
            const uint32_t kk = order_key(vv[e]);
            if (kk > thr) {
              sortbuf[atomicAdd(&n_gt, 1u)] = sort_key(kk, j4 + e);
            } else if (kk == thr && eq_total == need) {
              sortbuf[base_eq + atomicAdd(&n_eq, 1u)] = sort_key(kk, j4 + e);
            }
          }
        }
        if (eq_total > need) {
          // more equal scores than slots: the lowest-numbered ones, by an ordered scan
          __syncthreads();
          for (int j0 = 0; j0 < n; j0 += blockDim.x) {
            const int j = j0 + t;
            const bool eq = j < n && order_key(srow[j]) == thr;
            const unsigned bal = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) scratch[warp] = __popc(bal);
            __syncthreads();
            if (t < 32) {
              const int nw = blockDim.x / 32;
              uint32_t v = t < nw ? scratch[t] : 0u, incl = v;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (t >= o) incl += y;
              }
              if (t < nw) scratch[t] = incl - v;
              if (t == 31) scratch[kTopkThreads - 1] = incl;
            }
            __syncthreads();
            if (eq) {
              const uint32_t rank = eq_base + scratch[warp] + __popc(bal & ((1u << lane) - 1u));
              if (rank < need) sortbuf[base_eq + rank] = sort_key(thr, j);
            }
            __syncthreads();
            if (t == 0) eq_base += scratch[kTopkThreads - 1];
            __syncthreads();
            if (eq_base >= need) break;            // uniform: read after the barrier
          }
        }
      }
      __syncthreads();
      // bitonic sort of sortbuf[0 .. n_out) ascending (pad with all-ones)
      int len = 1;
      while (len < n_out) len <<= 1;
      for (int x = n_out + t; x < len; x += blockDim.x) sortbuf[x] = ~0ull;
      __syncthreads();
      for (int size = 2; size <= len; size <<= 1) {
        for (int st = size >> 1; st > 0; st >>= 1) {
          for (int x = t; x < len; x += blockDim.x) {
            const int y = x ^ st;
            if (y > x) {
              const bool up = (x & size) == 0;
              const unsigned long long a = sortbuf[x], c = sortbuf[y];
              if ((a > c) == up) {
                sortbuf[x] = c;
                sortbuf[y] = a;
              }
            }
          }
          __syncthreads();
        }
      }
      int32_t* irow = p.idx + (int64_t)(m.off_o + r) * topk;
      float* orow = p.score_out ? p.score_out + (int64_t)(m.off_o + r) * topk : nullptr;
      for (int x = t; x < topk; x += blockDim.x) {
        if (x < n_out) {
          const int j = (int)(uint32_t)sortbuf[x];
          irow[x] = j;
          if (orow) orow[x] = srow[j];
        } else {
          irow[x] = -1;
          if (orow) orow[x] = __int_as_float(0x7fc00000);
        }
      }
      __syncthreads();
    }
  }
}

template <typename T>
cudaError_t launch_scores_t(const IndexerParams& p, int num_sms, cudaStream_t stream) {
  const int smem = (p.heads * p.d + p.heads) * 4;
  cudaError_t e = cudaFuncSetAttribute(indexer_scores_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  indexer_scores_simt_kernel<T><<<num_sms * 4, kScoreThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_scores_simt(const IndexerParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream) {
  return dtype == THD_BF16 ? launch_scores_t<__nv_bfloat16>(p, num_sms, stream)
                           : launch_scores_t<__half>(p, num_sms, stream);
}

cudaError_t launch_indexer_topk(const IndexerParams& p, int num_sms, cudaStream_t stream) {
  indexer_topk_kernel<<<num_sms * 8, kTopkThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace thd
