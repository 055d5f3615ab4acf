// Internal declarations shared by the host API and the kernels of libthd_attn.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "thd_attn.h"

namespace thd {

// Words of the workspace header. The tile counter is word 0 (the persistent
// scheduler's claim counter); everything after it is sized by the plan.
// Words kHdrGroupStart .. kHdrGroupStart + kCostGroups hold the first pair index
// of each cost group (cost = KV tiles a pair visits; group 0 = costs 512..1023,
// group 1 = 256..511, ..., group 9 = cost 1, group 10 = cost 0), the last word
// being the pair count.
enum HeaderWord : int {
  kHdrCounter = 0, kHdrStatus = 1, kHdrNumPairs = 2, kHdrNumTiles = 3, kHdrGroupStart = 4,
  kHdrNumSplit = 16  // pairs whose KV range is split (partials merged by the combine kernel)
};
constexpr int kCostGroups = 11;
constexpr int kHeaderBytes = 128;
static_assert(kHdrGroupStart + kCostGroups + 1 <= kHdrNumSplit, "header words");
static_assert((kHdrNumSplit + 1) * 4 <= kHeaderBytes, "header words");

// KV split: when a launch has fewer than kSplitWaves waves of units, every pair
// visiting at least kMinSplitCost KV tiles is processed as two halves of its KV
// range whose partial results are merged afterwards. When the halves then leave a
// last, partial wave of units (and at least one full wave before it), the
// cheapest split pairs whose units would fill that wave are cut into kTailParts
// parts instead, so the end of the launch is filled with short units rather than
// leaving CTAs idle; only pairs of at least kMinTailCost tiles qualify.
// kMaxSmsForSizing bounds the SM count the workspace is sized for.
constexpr int kSplitWaves = 4;
constexpr int kMinSplitCost = 16;   // each half keeps >= 8 tiles to amortise a unit's fill and epilogue
constexpr int kTailParts = 8;
constexpr int kMinTailCost = 8 * kTailParts;
constexpr int kMaxSmsForSizing = 160;
// split pairs cut into kTailParts parts at most: the units of a last, partial wave
// number rest < CTAs <= kMaxSmsForSizing, which are ceil(rest / unit_heads) half
// entries of unit_heads units each, i.e. at most half as many pairs (rounded up)
__host__ __device__ constexpr int max_tail_pairs(int unit_heads) {
  return ((kMaxSmsForSizing + unit_heads - 1) / unit_heads + 1) / 2;
}

// Per-sequence record written by the setup kernel. `shift` is the causal shift:
// query row i sees keys j < len_k with j <= i + shift (mask 0 stores len_k, which
// lets every key through for any i >= 0); `lo_shift` the window's lower end:
// also j >= i + lo_shift (kNoLowerBound when unbounded). The last three words are
// written by the backward's key-axis setup only (zero elsewhere): the key group's
// member count (0 for a member that is not the group's first sequence), the
// group's key length (longest valid member), and the sequence's status bits.
struct SeqMeta {
  int32_t len_q, len_k, off_q, off_k, off_v, off_o, off_s, shift, lo_shift;
  int32_t group_n, group_len_k, bad;
};
static_assert(sizeof(SeqMeta) == 48, "SeqMeta is 48 bytes");
constexpr int32_t kNoLowerBound = -(1 << 30);

// A scheduled unit: rows [row0, row0 + rows_per_unit) of sequence b, for every
// query head. `split` = (i << 8) | parts: parts is 1 for a whole pair, else the
// pair's KV tile span [0, n) is processed in `parts` pieces and this entry covers
// [i n / parts, (i + 1) n / parts); `part` is the entry's slot in the
// partial-result buffers (-1 when whole).
struct PairRec {
  int32_t b, row0, split, part;
};
static_assert(sizeof(PairRec) == 16, "PairRec is 16 bytes");

// A pair whose KV range was split, for the combine kernel: where its rows are and
// its partial slots [slot0, slot0 + parts).
struct SplitRec {
  int32_t b, row0, slot0, parts;
};

constexpr int kCostBins = 1024;          // LPT buckets of the setup kernel's counting sort
constexpr int kSetupThreads = 1024;

struct SetupParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* off_q;
  const int32_t* off_k;
  const int32_t* off_v;
  const int32_t* off_o;
  const int32_t* off_s;
  const int8_t* mask;
  const int32_t* qco;       // may be null
  const int32_t* window;    // may be null
  int64_t cap_q, cap_k, cap_v, cap_o, cap_s;
  int32_t batch;
  int32_t rows_per_unit;    // rows (keys on the key axis) of one scheduled unit
  int32_t keys_per_tile;    // keys per KV tile (query rows per tile on the key axis)
  int32_t max_pairs;        // pairs before splitting
  int32_t h_q;
  int32_t key_axis;         // 0: units over query rows (cost = KV tiles); 1: over keys (cost = query tiles)
  int64_t max_len_k;        // > 0: a longer key sequence is a BAD_LENGTH data error
  int32_t unit_heads;       // heads each pair is scheduled for (h_q, or h_kv on the key axis)
  int32_t allow_split;      // KV split permitted (workspace holds the partial buffers)
  int32_t element_offsets;  // offsets are elements (x multiplier): divide by the token strides
  int64_t offset_multiplier;
  int64_t tok_stride[5];    // Q K V O Stats token strides (elements), for element offsets
  int32_t num_ctas;         // persistent CTAs of the attention kernel
  int32_t max_split;        // capacity of the split-pair table
  int32_t max_tail;         // split pairs that may be cut into kTailParts parts
  int32_t pair_cap;         // capacity of the pair list (scheduled entries)
  int32_t slot_cap;         // partial-result slots (split parts)
  // key axis of the backward: consecutive sequences with the same K and V offsets
  // read the same key rows (zigzag context-parallel chunks of one document) and
  // form one group whose dK/dV units sum over all of its members; K/V rows of
  // different groups must not overlap (THD_DEV_KEY_OVERLAP otherwise)
  int32_t group_keys = 0;
  uint32_t* header;
  SeqMeta* meta;
  int32_t* pair_base;       // [batch + 1]
  PairRec* pairs;           // [pair_cap]
  SplitRec* splits;         // [max_split]
};

// Arguments common to both attention kernels.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* stats;
  int64_t stride_tok[4];    // elements, Q K V O
  int64_t stride_head[4];
  int64_t stats_tok, stats_head;
  int32_t h_q, h_kv, d;
  float scale_log2;         // softmax_scale * log2(e)
  const uint32_t* header;
  uint32_t* counter;
  uint32_t* status;
  const SeqMeta* meta;
  const PairRec* pairs;
  const SplitRec* splits;
  float* part_o;            // [slots][h_q][rows_per_unit][d] normalised partial O
  float* part_lse;          // [slots][h_q][rows_per_unit] partial LSE, base 2
  int32_t rows_per_unit;
  int32_t test_stall;       // test hook: see THD_FLAG_TEST_STALL
  int32_t has_window;       // a window tensor was passed (some lo_shift may be bounded)
};

// Work id -> (pair index into the pair list, query head). Pairs are sorted by
// descending cost; inside one cost group the order is kv head, then pair, then
// query head of the kv group, so units that read the same K/V (same sequence and
// kv head) run close together in time and share it through L2.
__device__ __forceinline__ void work_to_unit(const uint32_t* header, uint32_t w, int h_q, int h_kv, int& pair,
                                             int& head) {
  const uint32_t grp = (uint32_t)(h_q / h_kv);
  int g = 0;
  while (g < kCostGroups - 1 && w >= header[kHdrGroupStart + g + 1] * (uint32_t)h_q) ++g;
  const uint32_t start = header[kHdrGroupStart + g];
  const uint32_t size = header[kHdrGroupStart + g + 1] - start;
  const uint32_t local = w - start * (uint32_t)h_q;
  const uint32_t per_kvh = size * grp;
  const uint32_t kvh = local / per_kvh;
  const uint32_t rem = local - kvh * per_kvh;
  pair = (int)(start + rem / grp);
  head = (int)(kvh * grp + rem % grp);
}

// Arguments of the backward kernels. Tensor index of the stride arrays:
// 0 Q, 1 K, 2 V, 3 O, 4 dO, 5 dQ, 6 dK, 7 dV.
struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* d_o;
  const float* stats;
  void* dq;
  void* dk;
  void* dv;
  int64_t stride_tok[8];
  int64_t stride_head[8];
  int64_t stats_tok, stats_head;
  int32_t h_q, h_kv, d;
  float scale;              // softmax_scale
  float scale_log2;         // softmax_scale * log2(e)
  // query-axis schedule (dQ units: rows_per_unit query rows x one query head)
  const uint32_t* header_q;
  uint32_t* counter_q;
  const PairRec* pairs_q;
  // key-axis schedule (dK/dV units: keys_per_unit keys x one kv head)
  const uint32_t* header_k;
  uint32_t* counter_k;
  const PairRec* pairs_k;
  uint32_t* status;
  const SeqMeta* meta;
  const int32_t* pair_base_q;   // [B + 1] first query-axis pair of each sequence (unsorted numbering)
  // (LSE * log2(e), D = <dO, O>) per query row, in 128-row blocks: row i of sequence b
  // and head h sits at ld_index(pair_base_q, b, i, h, h_q); each block is 1 KB
  float2* ld;
  int32_t rows_per_unit;
  int32_t keys_per_unit;
  int32_t has_window;
};

// Arguments of the indexer kernels (scores, then per-row top-k).
struct IndexerParams {
  const void* q;            // QI [rows, H, d]
  const void* k;            // KI [rows, d]
  const float* w;           // W [rows of QI, H]
  int32_t* idx;             // [rows, topk]
  float* score_out;         // [rows, topk] or null
  float* scores;            // workspace: score_row floats per output row
  int64_t q_tok, q_head, k_tok, w_tok;
  int64_t score_row;
  int32_t heads, d, topk;
  const uint32_t* header;
  uint32_t* counter;
  const PairRec* pairs;
  const SeqMeta* meta;
  uint32_t* status;
  // key-axis schedule (tensor-core scores: units of 128 keys)
  const uint32_t* header_k;
  uint32_t* counter_k;
  const PairRec* pairs_k;
};
cudaError_t launch_indexer_scores_simt(const IndexerParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream);
cudaError_t launch_indexer_topk(const IndexerParams& p, int num_sms, cudaStream_t stream);
constexpr int kIndexerRowsPerUnit = 128;
constexpr int kIndexerKeysPerUnit = 256;   // keys of a tensor-core score unit
constexpr int kIndexerMaxTopk = 2048;

// index of query row i (of sequence b) and head h in BwdParams::ld
__device__ __forceinline__ int64_t ld_index(const int32_t* pair_base_q, int b, int i, int h, int h_q) {
  return ((int64_t)(pair_base_q[b] + i / 128) * h_q + h) * 128 + (i & 127);
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_setup(const SetupParams& p, cudaStream_t stream);

cudaError_t launch_fwd_simt(const FwdParams& p, thd_dtype_t dtype, int rows_per_unit, int num_sms,
                            cudaStream_t stream);
int simt_rows_per_unit(int d);
cudaError_t launch_combine(const FwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream);
constexpr int kSimtKeysPerTile = 32;
// backward: preprocess (LSE and D per query row), then the dQ and dK/dV kernels
constexpr int kBwdRowsPerUnit = 128;   // query rows of a dQ unit
constexpr int kBwdKeysPerUnit = 128;   // keys of a dK/dV unit
cudaError_t launch_bwd_prep(const BwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_simt(const BwdParams& p, thd_dtype_t dtype, int num_sms, cudaStream_t stream);

}  // namespace thd

struct thd_attn_plan_s {
  thd_attn_desc_t desc;
  thd_kernel_t kernel;
  int32_t rows_per_unit;
  int32_t keys_per_tile;
  int32_t max_pairs;
  float scale;
  int64_t stats_tok, stats_head;
  int elem_bytes;
  size_t ws_bytes;
  int64_t ws_off[7];        // header, meta, pair_base, pairs, splits, part_o, part_lse
  int32_t allow_split;
  int32_t max_split;
  int32_t max_tail;
  int32_t pair_cap;         // pair list entries: max_pairs, or with splits every part of every pair
  int32_t slot_cap;         // partial-result slots
  // backward plans (thd_attn_plan_bwd)
  int32_t is_bwd;
  int64_t g_cap_rows[4];    // dO, dQ, dK, dV
  int64_t g_stride_tok[4];
  int64_t g_stride_head[4];
  int32_t max_pairs_k;      // key-axis pair capacity
  int64_t ws_off_b[4];      // key-axis header, pair_base, pairs; (LSE, D) rows
  // indexer plans (thd_indexer_plan): ws_off[0..3] as above, ws_off_b[0] the score rows
  int32_t is_indexer;
  thd_indexer_desc_t idesc;
  int64_t score_row;        // floats per output row in the score scratch
  // optional attention-kernel timing (thd_attn_profile_enable)
  int32_t prof_slots;
  int32_t prof_count;
  cudaEvent_t* prof_events; // 2 * prof_slots: start, stop pairs
};
