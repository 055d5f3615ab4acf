// Merge of split KV ranges: a pair whose key range the setup kernel cut into n
// parts (n = 2, or more at the end of a launch) left, for each part i, a normalised
// partial output O_i and a base-2 log-sum-exp L_i per (row, head) in the
// workspace. The row's result is the log-sum-exp weighted combination
//     M = max_i L_i,  w_i = 2^(L_i - M),  W = sum_i w_i,
//     O = sum_i w_i O_i / W,  LSE = (M + log2 W) * ln 2,
// which equals the softmax over the union of the key ranges; a row with no
// visible key in any part (every L_i = -inf) gets O = 0 and LSE = -inf. Only
// rows r < len_q of each pair are written, at the caller's O and Stats offsets.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace thd {

namespace {

template <typename T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<uint32_t*>(&lo);
  v.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float a, float b, float c, float d) {
  __half2 lo = __floats2half2_rn(a, b), hi = __floats2half2_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<uint32_t*>(&lo);
  v.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}

// One thread per (split pair, head, row, 4 consecutive elements of d): a warp reads
// 512 contiguous bytes of each partial row (float4 per lane) and many rows are in
// flight at once; the combine is bound by memory latency otherwise. d is a multiple
// of 4 (the tensor-core path serves d = 64 and 128), and O rows are 8-byte aligned.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(FwdParams p) {
  const uint32_t n_split = p.header[kHdrNumSplit];
  const int chunks = p.d >> 2;
  const int64_t rows_per_pair = (int64_t)p.h_q * p.rows_per_unit;
  const int64_t total = (int64_t)n_split * rows_per_pair * chunks;
  const int64_t threads = (int64_t)gridDim.x * blockDim.x;
  T* __restrict__ O = static_cast<T*>(p.o);
  for (int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; item < total; item += threads) {
    const int64_t idx = item / chunks;          // (pair, head, row)
    const int e = (int)(item - idx * chunks) * 4;
    const int part = (int)(idx / rows_per_pair);
    const int h = (int)((idx / p.rows_per_unit) % p.h_q);
    const int urow = (int)(idx % p.rows_per_unit);
    const SplitRec sr = p.splits[part];
    const SeqMeta m = p.meta[sr.b];
    const int r = sr.row0 + urow;
    if (r >= m.len_q) continue;
    // slot s holds rows [((s h_q + h) rows_per_unit + urow)]
    auto row_of = [&](int i) { return ((int64_t)(sr.slot0 + i) * p.h_q + h) * p.rows_per_unit + urow; };
    float mx = -INFINITY;
    for (int i = 0; i < sr.parts; ++i) mx = fmaxf(mx, p.part_lse[row_of(i)]);
    const bool dead = mx == -INFINITY;
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!dead) {
      for (int i = 0; i < sr.parts; ++i) {
        const int64_t ri = row_of(i);
        const float w = exp2f(p.part_lse[ri] - mx);
        const float4 a = *reinterpret_cast<const float4*>(p.part_o + ri * p.d + e);
        wsum += w;
        acc.x += w * a.x; acc.y += w * a.y; acc.z += w * a.z; acc.w += w * a.w;
      }
    }
    const float inv = dead ? 0.f : 1.f / wsum;
    T* orow = O + (int64_t)(m.off_o + r) * p.stride_tok[3] + (int64_t)h * p.stride_head[3];
    store4<T>(orow + e, acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (e == 0)
      p.stats[(int64_t)(m.off_s + r) * p.stats_tok + (int64_t)h * p.stats_head] =
          dead ? -INFINITY : (mx + log2f(wsum)) * 0.69314718055994530942f;
  }
}

}  // namespace

cudaError_t launch_combine(const FwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream) {
  const int blocks = num_sms * 8;
  switch (dtype) {
    case THD_BF16: combine_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(p); break;
    case THD_FP16: combine_kernel<__half><<<blocks, 256, 0, stream>>>(p); break;
    default: combine_kernel<float><<<blocks, 256, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace thd
