// Backward pass, SIMT kernels (fp32 arithmetic): the preprocess kernel used by
// every backward path, and general dQ and dK/dV kernels for fp32 inputs, head
// dims the tensor-core kernels do not take, and as a second GPU implementation
// for cross-checks.
//
// Gradients (ragged SDPA backward over the forward's metadata and Stats layouts,
// NVIDIA/cudnn-frontend PR #462, "What" / "Root cause"): with base-2 scores
// s2_ij = softmax_scale * log2(e) * <q_i, k_j> and LSE2_i = LSE_i * log2(e),
//   P_ij = 2^(s2_ij - LSE2_i) on visible keys, D_i = <dO_i, O_i>,
//   dS_ij = P_ij (<dO_i, v_j> - D_i),
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
//
// The preprocess kernel walks the query-axis schedule and stores (LSE2_i, D_i)
// per query row and head in the workspace. The dQ kernel claims query-axis units
// (rows x one query head) and walks their visible keys; the dK/dV kernel claims
// key-axis units (keys x one kv head) and walks, for every query head of the kv
// group, the query rows that see them, so dK and dV are complete sums with no
// atomics. Staged rows outside a sequence are zeros and contribute P = 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "convert.cuh"
#include "internal.h"

namespace thd {

namespace {

constexpr int kThreads = 128;
constexpr int kDPT = 32;   // head-dim elements per thread
constexpr int kBN = 32;    // keys staged per step (dQ kernel)
constexpr int kRB = 32;    // query rows staged per step (dK/dV kernel)

// sum over the TPR (<= 4) consecutive lanes that own one row
template <int TPR>
__device__ __forceinline__ float reduce_tpr(float a) {
  if (TPR >= 2) a += __shfl_xor_sync(0xffffffffu, a, 1);
  if (TPR >= 4) a += __shfl_xor_sync(0xffffffffu, a, 2);
  return a;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(BwdParams p) {
  const T* __restrict__ O = static_cast<const T*>(p.o);
  const T* __restrict__ G = static_cast<const T*>(p.d_o);
  const uint32_t num_tiles = p.header_q[kHdrNumTiles];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (uint32_t w = blockIdx.x; w < num_tiles; w += gridDim.x) {
    int pair_idx, h;
    work_to_unit(p.header_q, w, p.h_q, p.h_kv, pair_idx, h);
    const PairRec pr = p.pairs_q[pair_idx];
    const SeqMeta m = p.meta[pr.b];
    const int rows = min(p.rows_per_unit, m.len_q - pr.row0);
    for (int rr = warp; rr < rows; rr += kThreads / 32) {
      const int r = pr.row0 + rr;
      const T* orow = O + (int64_t)(m.off_o + r) * p.stride_tok[3] + (int64_t)h * p.stride_head[3];
      const T* grow = G + (int64_t)(m.off_o + r) * p.stride_tok[4] + (int64_t)h * p.stride_head[4];
      float acc = 0.f;
      for (int e = lane; e < p.d; e += 32) acc = fmaf(to_f32(orow[e]), to_f32(grow[e]), acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        const float lse = p.stats[(int64_t)(m.off_s + r) * p.stats_tok + (int64_t)h * p.stats_head];
        // a row whose LSE is -inf has no visible key: +inf turns every P of it into 0
        const float l2 = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
        p.ld[ld_index(p.pair_base_q, pr.b, r, h, p.h_q)] = make_float2(l2, acc);
      }
    }
  }
}

// ------------------------------------------------------------------------- dQ
template <typename T, int TPR>
__global__ void __launch_bounds__(kThreads) bwd_dq_simt_kernel(BwdParams p) {
  constexpr int ROWS = kThreads / TPR;
  constexpr int DMAX = kDPT * TPR;
  __shared__ float ks[kBN][DMAX];
  __shared__ float vs[kBN][DMAX];
  __shared__ uint32_t work_s;
  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ K = static_cast<const T*>(p.k);
  const T* __restrict__ V = static_cast<const T*>(p.v);
  const T* __restrict__ G = static_cast<const T*>(p.d_o);
  T* __restrict__ DQ = static_cast<T*>(p.dq);
  const int d = p.d;
  const int tid = threadIdx.x;
  const int lrow = tid / TPR;
  const int dbase = (tid % TPR) * kDPT;
  const uint32_t num_tiles = p.header_q[kHdrNumTiles];
  const int group = p.h_q / p.h_kv;

  for (;;) {
    if (tid == 0) work_s = atomicAdd(p.counter_q, 1u);
    __syncthreads();
    const uint32_t w = work_s;
    __syncthreads();
    if (w >= num_tiles) break;
    int pair_idx, h;
    work_to_unit(p.header_q, w, p.h_q, p.h_kv, pair_idx, h);
    const PairRec pr = p.pairs_q[pair_idx];
    const int g = h / group;
    const SeqMeta m = p.meta[pr.b];
    for (int sub = 0; sub < p.rows_per_unit; sub += ROWS) {
      if (pr.row0 + sub >= m.len_q) break;   // uniform across the block
      const int r = pr.row0 + sub + lrow;
      const bool live = r < m.len_q;
      float q[kDPT], go[kDPT], acc[kDPT];
#pragma unroll
      for (int e = 0; e < kDPT; ++e) q[e] = go[e] = acc[e] = 0.f;
      float l2 = INFINITY, dsum = 0.f;
      if (live) {
        const T* qrow = Q + (int64_t)(m.off_q + r) * p.stride_tok[0] + (int64_t)h * p.stride_head[0];
        const T* grow = G + (int64_t)(m.off_o + r) * p.stride_tok[4] + (int64_t)h * p.stride_head[4];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) {
            q[e] = to_f32(qrow[dbase + e]) * p.scale_log2;
            go[e] = to_f32(grow[dbase + e]);
          }
        const float2 ld = p.ld[ld_index(p.pair_base_q, pr.b, r, h, p.h_q)];
        l2 = ld.x;
        dsum = ld.y;
      }
      const int kmax_row = (int)max64(0, min64((int64_t)m.len_k, (int64_t)r + m.shift + 1));
      const int64_t kmin_row = (int64_t)r + m.lo_shift;
      const int64_t r_last = min64((int64_t)m.len_q, (int64_t)pr.row0 + sub + ROWS) - 1;
      const int kmax_unit = (int)max64(0, min64((int64_t)m.len_k, r_last + m.shift + 1));
      const int kmin_unit = (int)min64((int64_t)kmax_unit, max64(0, (int64_t)pr.row0 + sub + m.lo_shift));
      for (int j0 = kmin_unit / kBN * kBN; j0 < kmax_unit; j0 += kBN) {
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
#pragma unroll 4
        for (int jj = 0; jj < kBN; ++jj) {
          float s = 0.f, dp = 0.f;
#pragma unroll
          for (int e = 0; e < kDPT; ++e) {
            s = fmaf(q[e], ks[jj][dbase + e], s);
            dp = fmaf(go[e], vs[jj][dbase + e], dp);
          }
          s = reduce_tpr<TPR>(s);
          dp = reduce_tpr<TPR>(dp);
          const int j = j0 + jj;
          const bool vis = live && j < kmax_row && j >= kmin_row;
          const float pj = vis ? exp2f(s - l2) : 0.f;
          const float ds = pj * (dp - dsum);
#pragma unroll
          for (int e = 0; e < kDPT; ++e) acc[e] = fmaf(ds, ks[jj][dbase + e], acc[e]);
        }
        __syncthreads();
      }
      if (live) {
        T* dqrow = DQ + (int64_t)(m.off_q + r) * p.stride_tok[5] + (int64_t)h * p.stride_head[5];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) dqrow[dbase + e] = from_f32<T>(acc[e] * p.scale);
      }
    }
  }
}

// ---------------------------------------------------------------------- dK, dV
template <typename T, int TPR>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_simt_kernel(BwdParams p) {
  constexpr int KEYS = kThreads / TPR;
  constexpr int DMAX = kDPT * TPR;
  __shared__ float qs[kRB][DMAX];
  __shared__ float gs[kRB][DMAX];
  __shared__ float2 lds[kRB];
  __shared__ uint32_t work_s;
  const T* __restrict__ Q = static_cast<const T*>(p.q);
  const T* __restrict__ K = static_cast<const T*>(p.k);
  const T* __restrict__ V = static_cast<const T*>(p.v);
  const T* __restrict__ G = static_cast<const T*>(p.d_o);
  T* __restrict__ DK = static_cast<T*>(p.dk);
  T* __restrict__ DV = static_cast<T*>(p.dv);
  const int d = p.d;
  const int tid = threadIdx.x;
  const int lkey = tid / TPR;
  const int dbase = (tid % TPR) * kDPT;
  const uint32_t num_tiles = p.header_k[kHdrNumTiles];
  const int group = p.h_q / p.h_kv;

  for (;;) {
    if (tid == 0) work_s = atomicAdd(p.counter_k, 1u);
    __syncthreads();
    const uint32_t w = work_s;
    __syncthreads();
    if (w >= num_tiles) break;
    int pair_idx, g;
    work_to_unit(p.header_k, w, p.h_kv, p.h_kv, pair_idx, g);
    const PairRec pr = p.pairs_k[pair_idx];
    // the unit's key group: sequences pr.b .. pr.b + group_n - 1 read the same K/V
    // rows (keys < group_len_k); each adds the gradient of its own query rows
    const SeqMeta lead = p.meta[pr.b];
    const int n_mem = max(1, lead.group_n);
    for (int sub = 0; sub < p.keys_per_unit; sub += KEYS) {
      if (pr.row0 + sub >= lead.group_len_k) break;   // uniform across the block
      const int j = pr.row0 + sub + lkey;    // key inside the group
      const bool live = j < lead.group_len_k;
      const SeqMeta& m = lead;
      float kk[kDPT], vv[kDPT], dk[kDPT], dv[kDPT];
#pragma unroll
      for (int e = 0; e < kDPT; ++e) kk[e] = vv[e] = dk[e] = dv[e] = 0.f;
      if (live) {
        const T* krow = K + (int64_t)(m.off_k + j) * p.stride_tok[1] + (int64_t)g * p.stride_head[1];
        const T* vrow = V + (int64_t)(m.off_v + j) * p.stride_tok[2] + (int64_t)g * p.stride_head[2];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) {
            kk[e] = to_f32(krow[dbase + e]) * p.scale_log2;
            vv[e] = to_f32(vrow[dbase + e]);
          }
      }
      for (int mb = pr.b; mb < pr.b + n_mem; ++mb) {   // members of the key group
        const SeqMeta mm = p.meta[mb];
        const int64_t j_first = (int64_t)pr.row0 + sub;
        if (mm.bad != 0 || j_first >= mm.len_k) continue;   // uniform across the block
        const bool live_m = live && j < mm.len_k;
        // query rows that see any key of this pass: j - shift <= i <= j - lo_shift
        const int64_t j_last = min64((int64_t)mm.len_k, j_first + KEYS) - 1;
        const int i_lo = (int)min64((int64_t)mm.len_q, max64(0, j_first - (int64_t)mm.shift));
        const int i_hi = (int)max64((int64_t)i_lo, min64((int64_t)mm.len_q, j_last - (int64_t)mm.lo_shift + 1));
        for (int h = g * group; h < (g + 1) * group; ++h) {
          for (int i0 = i_lo; i0 < i_hi; i0 += kRB) {
            for (int idx = tid; idx < kRB * DMAX; idx += kThreads) {
              const int ii = idx / DMAX, e = idx % DMAX;
              const int i = i0 + ii;
              float qv = 0.f, gv = 0.f;
              if (i < i_hi && e < d) {
                qv = to_f32(Q[(int64_t)(mm.off_q + i) * p.stride_tok[0] + (int64_t)h * p.stride_head[0] + e]);
                gv = to_f32(G[(int64_t)(mm.off_o + i) * p.stride_tok[4] + (int64_t)h * p.stride_head[4] + e]);
              }
              qs[ii][e] = qv;
              gs[ii][e] = gv;
            }
            if (tid < kRB) {
              const int i = i0 + tid;
              lds[tid] = i < i_hi ? p.ld[ld_index(p.pair_base_q, mb, i, h, p.h_q)] : make_float2(INFINITY, 0.f);
            }
            __syncthreads();
  #pragma unroll 4
            for (int ii = 0; ii < kRB; ++ii) {
              float s = 0.f, dp = 0.f;
  #pragma unroll
              for (int e = 0; e < kDPT; ++e) {
                s = fmaf(kk[e], qs[ii][dbase + e], s);
                dp = fmaf(vv[e], gs[ii][dbase + e], dp);
              }
              s = reduce_tpr<TPR>(s);
              dp = reduce_tpr<TPR>(dp);
              const int64_t i = (int64_t)i0 + ii;
              const bool vis = live_m && i < i_hi && (int64_t)j <= i + mm.shift && (int64_t)j >= i + mm.lo_shift;
              const float2 ld = lds[ii];
              const float pj = vis ? exp2f(s - ld.x) : 0.f;
              const float ds = pj * (dp - ld.y);
  #pragma unroll
              for (int e = 0; e < kDPT; ++e) {
                dv[e] = fmaf(pj, gs[ii][dbase + e], dv[e]);
                dk[e] = fmaf(ds, qs[ii][dbase + e], dk[e]);
              }
            }
            __syncthreads();
          }
        }
      }
      if (live) {
        T* dkrow = DK + (int64_t)(m.off_k + j) * p.stride_tok[6] + (int64_t)g * p.stride_head[6];
        T* dvrow = DV + (int64_t)(m.off_v + j) * p.stride_tok[7] + (int64_t)g * p.stride_head[7];
#pragma unroll
        for (int e = 0; e < kDPT; ++e)
          if (dbase + e < d) {
            dkrow[dbase + e] = from_f32<T>(dk[e] * p.scale);
            dvrow[dbase + e] = from_f32<T>(dv[e]);
          }
      }
    }
  }
}

template <typename T, int TPR>
cudaError_t launch_simt_t(const BwdParams& p, int num_sms, cudaStream_t stream) {
  const int blocks = num_sms * 8;
  bwd_dq_simt_kernel<T, TPR><<<blocks, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dkdv_simt_kernel<T, TPR><<<blocks, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt_d(const BwdParams& p, int num_sms, cudaStream_t stream) {
  if (p.d <= kDPT) return launch_simt_t<T, 1>(p, num_sms, stream);
  if (p.d <= 2 * kDPT) return launch_simt_t<T, 2>(p, num_sms, stream);
  return launch_simt_t<T, 4>(p, num_sms, stream);
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream) {
  const int blocks = num_sms * 8;
  switch (dtype) {
    case THD_BF16: bwd_prep_kernel<__nv_bfloat16><<<blocks, kThreads, 0, stream>>>(p); break;
    case THD_FP16: bwd_prep_kernel<__half><<<blocks, kThreads, 0, stream>>>(p); break;
    default: bwd_prep_kernel<float><<<blocks, kThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream) {
  switch (dtype) {
    case THD_BF16: return launch_simt_d<__nv_bfloat16>(p, num_sms, stream);
    case THD_FP16: return launch_simt_d<__half>(p, num_sms, stream);
    default: return launch_simt_d<float>(p, num_sms, stream);
  }
}

}  // namespace thd
