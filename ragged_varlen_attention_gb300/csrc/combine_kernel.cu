// Merge of split KV ranges: a pair whose key range the setup kernel split in two
// left, for each half h in {0, 1}, a normalised partial output O_h and a base-2
// log-sum-exp L_h per (row, head) in the workspace. The row's result is the
// log-sum-exp weighted combination
//     M = max(L_0, L_1),  w_h = 2^(L_h - M),  W = w_0 + w_1,
//     O = (w_0 O_0 + w_1 O_1) / W,  LSE = (M + log2 W) * ln 2,
// which equals the softmax over the union of the two key ranges; a row with no
// visible key in either half (both L_h = -inf) gets O = 0 and LSE = -inf. Only
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
    const int64_t base0 = ((int64_t)(2 * part) * p.h_q + h) * p.rows_per_unit + urow;
    const int64_t base1 = ((int64_t)(2 * part + 1) * p.h_q + h) * p.rows_per_unit + urow;
    const float l0 = p.part_lse[base0], l1 = p.part_lse[base1];
    const float4 a = *reinterpret_cast<const float4*>(p.part_o + base0 * p.d + e);
    const float4 b = *reinterpret_cast<const float4*>(p.part_o + base1 * p.d + e);
    const float mx = fmaxf(l0, l1);
    const bool dead = mx == -INFINITY;
    const float w0 = dead ? 0.f : exp2f(l0 - mx), w1 = dead ? 0.f : exp2f(l1 - mx);
    const float wsum = w0 + w1;
    const float inv = dead ? 0.f : 1.f / wsum;
    T* orow = O + (int64_t)(m.off_o + r) * p.stride_tok[3] + (int64_t)h * p.stride_head[3];
    store4<T>(orow + e, (w0 * a.x + w1 * b.x) * inv, (w0 * a.y + w1 * b.y) * inv, (w0 * a.z + w1 * b.z) * inv,
              (w0 * a.w + w1 * b.w) * inv);
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
