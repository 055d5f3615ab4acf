// Pieces shared by the tensor-core kernels: bounded mbarrier waits, 16-bit
// packing, and TMA descriptors over [rows, heads, d] views.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace thd {
namespace tc {

constexpr uint64_t kWaitLimitNs = 4000000000ull;

struct Sync {
  uint32_t bar0;               // shared address of barrier 0
  volatile int* abort_flag;
  uint32_t* status;
  int spins = 96;              // non-blocking probes before the sleep-hinted waits
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  // bounded wait for the phase of `parity` on barrier i; false on abort/timeout
  __device__ __forceinline__ bool wait(int i, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) const {
    const uint32_t b = bar(i);
    // short spin of non-blocking probes (wake-up latency matters on the critical
    // path), then sleep-hinted blocking tries so long waits leave the issue slots
    // to other warps
    for (int k = 0; k < spins; ++k)
      if (ptx::mbar_test_wait(b, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
      if (ptx::mbar_try_wait_sleep(b, parity, 20000u)) return true;
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, (uint32_t)THD_DEV_WAIT_TIMEOUT);
        return false;
      }
    }
  }
  // every lane waits; the outcome is made warp-uniform (an abort seen by one lane
  // stops the whole warp) so the warp never diverges around a warp-wide operation
  __device__ __forceinline__ bool wait_warp(int i, uint32_t parity) const {
    const bool r = wait(i, parity);
    return __all_sync(0xffffffffu, r);
  }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

}  // namespace tc

namespace tc_host {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// [rows, heads, d] view, box = 64 d-elements x 1 head x box_rows rows, 128-byte
// swizzle; rows past `rows` read as zeros
inline bool encode_view(CUtensorMap* map, const void* base, bool bf16, int d, int64_t heads, int64_t rows,
                 int64_t stride_head, int64_t stride_tok, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)(stride_head * 2), (cuuint64_t)(stride_tok * 2)};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// general tiled map: `rank` dims (innermost first) with byte strides of the outer
// dims, a box, and a swizzle mode; rows past a dim read as zeros
inline bool encode_tiled(CUtensorMap* map, const void* base, CUtensorMapDataType type, int rank,
                         const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                         CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tc_host
}  // namespace thd
