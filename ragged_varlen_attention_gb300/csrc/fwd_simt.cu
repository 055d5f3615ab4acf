// SIMT forward kernel: the general path for fp32 inputs and for head dims the
// tensor-core kernel does not take (any d <= 128), and a second, independent
// GPU implementation for cross-checks. fp32 arithmetic throughout.
//
// Persistent blocks claim scheduled units from the workspace tile counter
// (cudnn-frontend PR #462, "Root cause": tile_id = atomicAdd(counter, 1), retire
// once tile_id >= num_tiles). A unit is `rows` query rows of one sequence and one
// query head, processed kThreads / TPR rows at a time; each row is owned by TPR threads (TPR = 1 for d <= 64, 2 for
// d <= 128), each holding a 64-wide slice of q and of the output accumulator in
// registers. Keys are staged in shared memory 32 at a time as fp32; key rows past
// len_k are staged as zeros, so pad contents (NaN included) never reach the math
// (cuDNN-frontend issue on THD offsets: pad slots have no initialization
// guarantee). Online softmax in base 2; rows with no visible key store O = 0 and
// LSE = -inf; only rows r < len_q are stored.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "convert.cuh"
#include "internal.h"

namespace thd {

namespace {

constexpr int kThreads = 128;
constexpr int kBN = kSimtKeysPerTile;
constexpr int kDPT = 64;  // head-dim elements per thread

template <typename T, int TPR>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdParams p, int rows_per_unit) {
  constexpr int ROWS = kThreads / TPR;
  constexpr int DMAX = kDPT * TPR;
  __shared__ float ks[kBN][DMAX];
  __shared__ float vs[kBN][DMAX];
  __shared__ uint32_t work_s;

  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ K = static_cast<const T*>(p.k);
  const T* __restrict__ V = static_cast<const T*>(p.v);
  T* __restrict__ O = static_cast<T*>(p.o);
  const int d = p.d;
  const int tid = threadIdx.x;
  const int lrow = tid / TPR;        // row within the unit
  const int part = tid % TPR;        // which 64-wide slice of d
  const int dbase = part * kDPT;
  const uint32_t num_tiles = p.header[kHdrNumTiles];
  const int group = p.h_q / p.h_kv;

  for (;;) {
    if (tid == 0) work_s = atomicAdd(p.counter, 1u);
    __syncthreads();
    const uint32_t w = work_s;
    __syncthreads();
    if (w >= num_tiles) break;
    int pair_idx, h;
    work_to_unit(p.header, w, p.h_q, p.h_kv, pair_idx, h);
    const PairRec pr = p.pairs[pair_idx];
    const int g = h / group;
    const SeqMeta m = p.meta[pr.b];
    for (int sub = 0; sub < rows_per_unit; sub += ROWS) {
      if (pr.row0 + sub >= m.len_q) break;          // uniform across the block
      const int r = pr.row0 + sub + lrow;           // row inside the sequence
      const bool row_live = r < m.len_q;

      float q[kDPT], acc[kDPT];
#pragma unroll
      for (int e = 0; e < kDPT; ++e) {
        acc[e] = 0.f;
        q[e] = 0.f;
      }
      if (row_live) {
        const T* qrow = Q + (int64_t)(m.off_q + r) * p.stride_tok[0] + (int64_t)h * p.stride_head[0];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) q[e] = to_f32(qrow[dbase + e]) * p.scale_log2;
      }
      float mrow = -INFINITY, lrow_sum = 0.f;
      // keys this row may see: j < kmax_row
      const int64_t kmax_row64 = min64((int64_t)m.len_k, (int64_t)r + m.shift + 1);
      const int kmax_row = (int)max64(0, kmax_row64);
      // lowest key this row may see (window), and the key range any row of the block may see
      const int64_t kmin_row = (int64_t)r + m.lo_shift;
      const int64_t r_last = min64((int64_t)m.len_q, (int64_t)pr.row0 + sub + ROWS) - 1;
      const int kmax_unit = (int)max64(0, min64((int64_t)m.len_k, r_last + m.shift + 1));
      const int kmin_unit = (int)min64((int64_t)kmax_unit, max64(0, (int64_t)pr.row0 + sub + m.lo_shift));

      for (int j0 = kmin_unit / kBN * kBN; j0 < kmax_unit; j0 += kBN) {
        // stage K/V rows j0 .. j0+kBN-1 (zeros past len_k)
        for (int idx = tid; idx < kBN * DMAX; idx += kThreads) {
          const int jj = idx / DMAX, e = idx % DMAX;
          const int j = j0 + jj;
          float kv = 0.f, vv = 0.f;
          if (j < m.len_k && e < d) {
            kv = to_f32(K[(int64_t)(m.off_k + j) * p.stride_tok[1] + (int64_t)g * p.stride_head[1] + e]);
            vv = to_f32(V[(int64_t)(m.off_v + j) * p.stride_tok[2] + (int64_t)g * p.stride_head[2] + e]);
          }
          ks[jj][e] = kv;
          vs[jj][e] = vv;
        }
        __syncthreads();
        float s[kBN];
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kBN; ++jj) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < kDPT; ++e) a = fmaf(q[e], ks[jj][dbase + e], a);
          if (TPR == 2) a += __shfl_xor_sync(0xffffffffu, a, 1);
          s[jj] = (j0 + jj < kmax_row && j0 + jj >= kmin_row) ? a : -INFINITY;
          tmax = fmaxf(tmax, s[jj]);
        }
        const float mnew = fmaxf(mrow, tmax);
        if (mnew != -INFINITY) {
          const float alpha = exp2f(mrow - mnew);  // mrow = -inf -> 0
          lrow_sum *= alpha;
#pragma unroll
          for (int e = 0; e < kDPT; ++e) acc[e] *= alpha;
#pragma unroll
          for (int jj = 0; jj < kBN; ++jj) {
            const float pj = exp2f(s[jj] - mnew);
            lrow_sum += pj;
#pragma unroll
            for (int e = 0; e < kDPT; ++e) acc[e] = fmaf(pj, vs[jj][dbase + e], acc[e]);
          }
          mrow = mnew;
        }
        __syncthreads();
      }

      if (row_live) {
        const bool live = lrow_sum > 0.f;
        const float inv = live ? 1.f / lrow_sum : 0.f;
        T* orow = O + (int64_t)(m.off_o + r) * p.stride_tok[3] + (int64_t)h * p.stride_head[3];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) orow[dbase + e] = from_f32<T>(acc[e] * inv);
        if (part == 0) {
          const float lse = live ? (mrow + log2f(lrow_sum)) * 0.69314718055994530942f : -INFINITY;
          p.stats[(int64_t)(m.off_s + r) * p.stats_tok + (int64_t)h * p.stats_head] = lse;
        }
      }
    }
  }
}

template <typename T>
cudaError_t launch_t(const FwdParams& p, int rows_per_unit, int num_sms, cudaStream_t stream) {
  const int blocks = num_sms * 8;
  if (p.d <= kDPT) fwd_simt_kernel<T, 1><<<blocks, kThreads, 0, stream>>>(p, rows_per_unit);
  else fwd_simt_kernel<T, 2><<<blocks, kThreads, 0, stream>>>(p, rows_per_unit);
  return cudaGetLastError();
}

}  // namespace

int simt_rows_per_unit(int d) { return d <= kDPT ? kThreads : kThreads / 2; }

cudaError_t launch_fwd_simt(const FwdParams& p, thd_dtype_t dtype, int rows_per_unit, int num_sms,
                            cudaStream_t stream) {
  switch (dtype) {
    case THD_BF16: return launch_t<__nv_bfloat16>(p, rows_per_unit, num_sms, stream);
    case THD_FP16: return launch_t<__half>(p, rows_per_unit, num_sms, stream);
    default: return launch_t<float>(p, rows_per_unit, num_sms, stream);
  }
}

}  // namespace thd
