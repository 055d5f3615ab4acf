// Indexer top-k kernels: a SIMT score kernel (any H <= 128, d <= 128; fp32
// arithmetic) and the per-row top-k selection shared by every score path.
//
// Scores (lightning-indexer form, see thd_indexer_topk in thd_attn.h):
// I_ij = sum_h w_ih * max(0, <q_ih, k_j>) for the visible prefix j < kmax_i of
// each row (the attention forward's mask policy and q_causal_offset; Megatron-LM
// PR #14 "fix(dsa): align packed-CP indexer causal masks"). Each output row owns a
// float32 row of the workspace; key j's score sits at column j.
//
// Top-k (one CTA per row at a time, persistent over the scheduled 128-row units):
// scores are mapped to order-preserving unsigned keys, the k-th largest key is
// found by a three-pass radix select over 11 + 11 + 10 bits (shared-memory
// histograms), every key above that threshold and the lowest-numbered keys equal
// to it are gathered (exactly k), and the k entries are sorted by descending score
// then ascending key number with a bitonic sort in shared memory. Rows with at
// most k visible keys skip the select and sort all of them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "convert.cuh"
#include "internal.h"

namespace thd {

namespace {

constexpr int kScoreThreads = 256;
constexpr int kTopkThreads = 512;

// ------------------------------------------------------------------- scores (SIMT)
template <typename T>
__global__ void __launch_bounds__(kScoreThreads) indexer_scores_simt_kernel(IndexerParams p) {
  extern __shared__ float qs[];              // [H][d] of the current row, then w [H]
  const int H = p.heads, d = p.d;
  float* ws = qs + H * d;
  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ K = static_cast<const T*>(p.k);
  const uint32_t num_tiles = p.header[kHdrNumTiles];
  for (uint32_t w = blockIdx.x; w < num_tiles; w += gridDim.x) {
    int pair, head;
    work_to_unit(p.header, w, 1, 1, pair, head);
    const PairRec pr = p.pairs[pair];
    const SeqMeta m = p.meta[pr.b];
    const int rows = min(kIndexerRowsPerUnit, m.len_q - pr.row0);
    for (int rr = 0; rr < rows; ++rr) {
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

__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(IndexerParams p) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t scratch[kTopkThreads];
  __shared__ unsigned long long sortbuf[kIndexerMaxTopk];
  __shared__ int sel_bin;
  __shared__ uint32_t n_sel, eq_base;
  const uint32_t num_tiles = p.header[kHdrNumTiles];
  const int t = threadIdx.x;
  const int topk = p.topk;
  for (uint32_t w = blockIdx.x; w < num_tiles; w += gridDim.x) {
    int pair, head;
    work_to_unit(p.header, w, 1, 1, pair, head);
    const PairRec pr = p.pairs[pair];
    const SeqMeta m = p.meta[pr.b];
    const int rows = min(kIndexerRowsPerUnit, m.len_q - pr.row0);
    for (int rr = 0; rr < rows; ++rr) {
      const int r = pr.row0 + rr;
      const int n = (int)max64(0, min64((int64_t)m.len_k, (int64_t)r + m.shift + 1));
      const float* srow = p.scores + (int64_t)(m.off_o + r) * p.score_row;
      int n_out = min(n, topk);
      if (t == 0) n_sel = 0;
      __syncthreads();
      if (n <= topk) {
        for (int j = t; j < n; j += blockDim.x)
          sortbuf[j] = ((unsigned long long)(0xffffffffu - order_key(srow[j])) << 32) | (uint32_t)j;
      } else {
        // radix select of the topk-th largest key: bits 31..21, 20..10, 9..0
        uint32_t prefix = 0, need = (uint32_t)topk;
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
          const int nb = 1 << widths[pass];
          for (int b = t; b < 2048; b += blockDim.x) hist[b] = 0;
          __syncthreads();
          const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (shifts[pass] + widths[pass]));
          for (int j = t; j < n; j += blockDim.x) {
            const uint32_t kk = order_key(srow[j]);
            if ((kk & hi_mask) == prefix) atomicAdd(&hist[(kk >> shifts[pass]) & (nb - 1)], 1u);
          }
          __syncthreads();
          suffix_sums(hist, nb, scratch);
          const int b = find_bin(hist, nb, need, &sel_bin);
          const uint32_t above = b + 1 < nb ? hist[b + 1] : 0u;
          need -= above;
          prefix |= (uint32_t)b << shifts[pass];
          __syncthreads();
        }
        // prefix is the threshold key; `need` elements equal to it are taken, the
        // lowest-numbered ones, after every element above it
        const uint32_t thr = prefix;
        if (t == 0) eq_base = 0;
        __syncthreads();
        for (int j0 = 0; j0 < n; j0 += blockDim.x) {
          const int j = j0 + t;
          uint32_t kk = 0;
          bool gt = false, eq = false;
          if (j < n) {
            kk = order_key(srow[j]);
            gt = kk > thr;
            eq = kk == thr;
          }
          if (gt) {
            const uint32_t slot = atomicAdd(&n_sel, 1u);
            sortbuf[slot] = ((unsigned long long)(0xffffffffu - kk) << 32) | (uint32_t)j;
          }
          // rank of this equal element in index order within the chunk
          const unsigned bal = __ballot_sync(0xffffffffu, eq);
          const int lane = t & 31, warp = t >> 5;
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
            if (t == 31) scratch[kTopkThreads - 1] = incl;   // chunk total
          }
          __syncthreads();
          if (eq) {
            const uint32_t rank = eq_base + scratch[warp] + __popc(bal & ((1u << lane) - 1u));
            if (rank < need) sortbuf[(uint32_t)topk - need + rank] = ((unsigned long long)(0xffffffffu - kk) << 32) | (uint32_t)j;
          }
          __syncthreads();
          if (t == 0) eq_base += scratch[kTopkThreads - 1];
          __syncthreads();
        }
      }
      __syncthreads();
      // bitonic sort of sortbuf[0 .. n_out) ascending (pad with all-ones)
      int len = 1;
      while (len < n_out) len <<= 1;
      for (int x = n_out + t; x < len; x += blockDim.x) sortbuf[x] = ~0ull;
      __syncthreads();
      for (int size = 2; size <= len; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int x = t; x < len; x += blockDim.x) {
            const int y = x ^ stride;
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
          const unsigned long long e = sortbuf[x];
          const int j = (int)(uint32_t)e;
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
  indexer_topk_kernel<<<num_sms * 2, kTopkThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace thd
