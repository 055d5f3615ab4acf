// tcgen05 forward kernel (placeholder until the tensor-core path lands).
#include "tc_launch.h"

namespace thd {

bool tc_kernel_available() { return false; }
int tc_rows_per_unit() { return 256; }
int tc_keys_per_tile() { return 128; }
cudaError_t launch_fwd_tc(const FwdParams&, const thd_attn_desc_t&, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace thd
