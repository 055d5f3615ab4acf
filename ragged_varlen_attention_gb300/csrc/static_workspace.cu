// thd_attn_fwd_static_ws: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they
// run attention: code executing while a stream is being captured into a CUDA
// graph, plugins hosted by a runtime that owns all device memory and forbids
// side allocations, and latency-critical serving loops where an allocation's
// implicit device synchronisation is not acceptable. This entry point takes no
// workspace argument. Its scratch lives in `g_static_workspace`, a file-scope
// device array of kStaticWorkspaceBytes that every GPU which loads this library
// holds until the process exits.
//
// In host code `g_static_workspace` names a host-side stand-in, not a device
// address, so it is never passed to a kernel directly: the first call on each
// device (with that device current) resolves the array's device address with
// cudaGetSymbolAddress and caches it. Make that first call before any stream
// capture begins.
//
// Every call on a device shares the one array, and the array keeps whatever the
// last call left in it. The setup kernel rewrites every word the attention
// kernel reads (header, metadata, tile list, and the tile counter, which it
// zeroes) before the attention kernel starts, so no clearing is needed between
// calls. Calls whose kernels overlap on the GPU (for example, on two streams
// without ordering between them) race on the array and must not be made.
#include <atomic>
#include <cstring>

#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of the array per device. Two host threads making their first
// call on a device at once may both resolve it; they store the same value.
std::atomic<void*> g_device_address[kMaxDevices];

// The array's device address on the current device (resolved once per device).
thd_status_t static_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return THD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return THD_ERR_CUDA;
  void* ptr = g_device_address[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return THD_ERR_CUDA;
    g_device_address[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return THD_OK;
}

}  // namespace

extern "C" {

size_t thd_attn_static_workspace_capacity(void) { return kStaticWorkspaceBytes; }

thd_status_t thd_attn_fwd_static_ws(thd_attn_plan_t plan, const void* q, const void* k, const void* v,
                                    void* o, float* stats, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_kv, const int32_t* off_q, const int32_t* off_k,
                                    const int32_t* off_v, const int32_t* off_o, const int32_t* off_s,
                                    const int8_t* mask_type, const int32_t* q_causal_offset, void* stream) {
  // only forward plans run here, whatever their workspace size
  if (!plan || plan->is_bwd || plan->is_indexer) return THD_ERR_INVALID_ARG;
  if (plan->ws_bytes > kStaticWorkspaceBytes) return THD_ERR_WORKSPACE;
  void* ws = nullptr;
  const thd_status_t st = static_address(&ws);
  if (st != THD_OK) return st;
  return thd_attn_fwd(plan, q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_v, off_o, off_s,
                      mask_type, q_causal_offset, ws, stream);
}

thd_status_t thd_attn_static_read_status(thd_attn_plan_t plan, uint32_t* host_out, void* stream) {
  if (!plan || !host_out || plan->is_bwd || plan->is_indexer) return THD_ERR_INVALID_ARG;
  void* ws = nullptr;
  const thd_status_t st = static_address(&ws);
  if (st != THD_OK) return st;
  return thd_attn_read_status(plan, ws, host_out, stream);
}

}  // extern "C"
