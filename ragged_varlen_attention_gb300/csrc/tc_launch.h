// Interface of the tcgen05 (tensor-core, TMEM, TMA) kernels: forward, backward and indexer scores.
#pragma once

#include "internal.h"

namespace thd {

bool tc_kernel_available();
int tc_rows_per_unit();   // query rows of one scheduled unit (two 128-row sub-tiles)
int tc_keys_per_tile();   // keys per KV tile
int tc_grid_size(int num_sms, int max_pairs, int h_q);  // persistent CTAs launched
// Encodes the TMA descriptors for Q/K/V from the plan's strides and launches the
// persistent kernel. Returns cudaErrorNotSupported when the descriptors cannot
// be encoded for these pointers/strides.
cudaError_t launch_fwd_tc(const FwdParams& p, const thd_attn_desc_t& desc, int max_pairs, int num_sms,
                          cudaStream_t stream);

// Backward: encodes TMA descriptors for Q, K, V and dO and launches the dQ and
// dK/dV kernels (after the setup and preprocess kernels). g_* index 0..3 = dO,
// dQ, dK, dV. Returns cudaErrorNotSupported when a descriptor cannot be encoded.
cudaError_t launch_bwd_tc(const BwdParams& p, const thd_attn_desc_t& desc, const int64_t g_cap[4],
                          const int64_t g_stok[4], const int64_t g_shead[4], int max_q, int max_k, int num_sms,
                          cudaStream_t stream);

// Indexer scores on the tensor cores: units of 128 keys (key-axis schedule in
// p.header_k), H in {4, 8, 16, 32, 64}, d in {64, 128}. cudaErrorNotSupported when
// the shape or a descriptor is not served.
bool indexer_tc_applicable(const thd_indexer_desc_t& d);
cudaError_t launch_indexer_scores_tc(const IndexerParams& p, const thd_indexer_desc_t& desc, int max_pairs_k,
                                     int num_sms, cudaStream_t stream);

}  // namespace thd
