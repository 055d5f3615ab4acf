// Host side of the C ABI declared in include/thd_attn.h: descriptor validation,
// capacity checks by the all-axes span rule (cudnn-frontend PR #462, "The fix"),
// kernel selection, workspace layouts, and the asynchronous enqueue of the
// forward, backward and indexer top-k passes.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "internal.h"
#include "tc_launch.h"

namespace {

constexpr int64_t kAlign = 256;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int elem_bytes(thd_dtype_t t) { return t == THD_FP32 ? 4 : 2; }

int num_sms_of_current_device() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

float scale_of(const thd_attn_desc_t& d) {
  return std::isnan(d.softmax_scale) ? 1.0f / std::sqrt((float)d.d) : d.softmax_scale;
}

// an indexer plan whose calls build a key-axis schedule (tensor-core scores)
bool indexer_uses_key_axis(const thd_attn_plan_s* plan) {
  return plan->is_indexer && plan->kernel == THD_KERNEL_TCGEN05 && plan->idesc.cap_rows_q > 0 &&
         plan->idesc.cap_rows_k > 0;
}

bool tc_applicable(const thd_attn_desc_t& d, float scale) {
  if (!thd::tc_kernel_available()) return false;
  if (!(scale > 0.f)) return false;  // the softmax takes the row max of unscaled scores
  if (d.dtype != THD_BF16 && d.dtype != THD_FP16) return false;
  if (d.d != 64 && d.d != 128) return false;
  const int eb = elem_bytes(d.dtype);
  for (int i = 0; i < 3; ++i) {  // Q, K, V go through TMA: 16-byte strides, < 2^31 rows
    if ((d.stride_tok[i] * eb) % 16 != 0 || (d.stride_head[i] * eb) % 16 != 0) return false;
    if (d.stride_tok[i] <= 0 || d.stride_head[i] <= 0) return false;
    if (d.cap_rows[i] >= (int64_t(1) << 31)) return false;
  }
  if ((d.stride_tok[3] * eb) % 16 != 0 || (d.stride_head[3] * eb) % 16 != 0) return false;
  return true;
}

}  // namespace

extern "C" {

int64_t thd_attn_view_span_bytes(int64_t rows, int64_t heads, int64_t d, int64_t stride_tok,
                                 int64_t stride_head, int64_t elem) {
  if (rows <= 0 || heads <= 0 || d <= 0) return 0;
  return ((rows - 1) * stride_tok + (heads - 1) * stride_head + (d - 1) + 1) * elem;
}

const char* thd_attn_status_string(thd_status_t s) {
  switch (s) {
    case THD_OK: return "THD_OK";
    case THD_ERR_INVALID_ARG: return "THD_ERR_INVALID_ARG";
    case THD_ERR_UNSUPPORTED: return "THD_ERR_UNSUPPORTED";
    case THD_ERR_ALIGNMENT: return "THD_ERR_ALIGNMENT";
    case THD_ERR_CAPACITY: return "THD_ERR_CAPACITY";
    case THD_ERR_WORKSPACE: return "THD_ERR_WORKSPACE";
    case THD_ERR_CUDA: return "THD_ERR_CUDA";
  }
  return "THD_ERR_UNKNOWN";
}

thd_status_t thd_attn_plan(thd_attn_plan_t* out, const thd_attn_desc_t* desc, size_t* ws_bytes) {
  if (!out || !desc || !ws_bytes) return THD_ERR_INVALID_ARG;
  *out = nullptr;
  const thd_attn_desc_t& d = *desc;
  if (d.dtype != THD_BF16 && d.dtype != THD_FP16 && d.dtype != THD_FP32) return THD_ERR_INVALID_ARG;
  if (d.batch < 0 || d.h_q < 1 || d.h_kv < 1 || d.h_q % d.h_kv != 0) return THD_ERR_INVALID_ARG;
  if (d.d < 1) return THD_ERR_INVALID_ARG;
  if (d.d > 128) return THD_ERR_UNSUPPORTED;
  if (d.stats_layout != THD_STATS_TOKEN_MAJOR && d.stats_layout != THD_STATS_HEAD_MAJOR)
    return THD_ERR_INVALID_ARG;
  if (d.kernel != THD_KERNEL_AUTO && d.kernel != THD_KERNEL_SIMT && d.kernel != THD_KERNEL_TCGEN05)
    return THD_ERR_INVALID_ARG;
  if (d.cap_rows_stats < 0 || d.cap_rows_stats >= (int64_t(1) << 31)) return THD_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {
    if (d.cap_rows[i] < 0 || d.cap_rows[i] >= (int64_t(1) << 31)) return THD_ERR_INVALID_ARG;
    if (d.stride_tok[i] < 0 || d.stride_head[i] < 0 || d.bytes[i] < 0) return THD_ERR_INVALID_ARG;
  }
  if (d.offset_multiplier < 0) return THD_ERR_INVALID_ARG;
  if (d.flags & THD_FLAG_ELEMENT_OFFSETS) {
    // element offsets are divided by the token strides on the device
    for (int i = 0; i < 4; ++i)
      if (d.stride_tok[i] <= 0) return THD_ERR_INVALID_ARG;
  }
  float scale = d.softmax_scale;
  if (std::isnan(scale)) scale = 1.0f / std::sqrt((float)d.d);
  if (!std::isfinite(scale)) return THD_ERR_INVALID_ARG;

  // capacity: the all-axes span of each declared view must fit its allocation
  const int eb = elem_bytes(d.dtype);
  const int64_t heads[4] = {d.h_q, d.h_kv, d.h_kv, d.h_q};
  for (int i = 0; i < 4; ++i) {
    if (d.bytes[i] == 0) continue;
    const int64_t span =
        thd_attn_view_span_bytes(d.cap_rows[i], heads[i], d.d, d.stride_tok[i], d.stride_head[i], eb);
    if (span > d.bytes[i]) return THD_ERR_CAPACITY;
  }

  thd_kernel_t kernel;
  if (d.kernel == THD_KERNEL_SIMT) {
    kernel = THD_KERNEL_SIMT;
  } else if (d.kernel == THD_KERNEL_TCGEN05) {
    if (!tc_applicable(d, scale)) return THD_ERR_UNSUPPORTED;
    kernel = THD_KERNEL_TCGEN05;
  } else {
    kernel = tc_applicable(d, scale) ? THD_KERNEL_TCGEN05 : THD_KERNEL_SIMT;
  }

  auto* p = new (std::nothrow) thd_attn_plan_s;
  if (!p) return THD_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->desc = d;
  p->kernel = kernel;
  p->scale = scale;
  p->elem_bytes = eb;
  if (kernel == THD_KERNEL_TCGEN05) {
    p->rows_per_unit = thd::tc_rows_per_unit();
    p->keys_per_tile = thd::tc_keys_per_tile();
  } else {
    p->rows_per_unit = thd::simt_rows_per_unit(d.d);
    p->keys_per_tile = thd::kSimtKeysPerTile;
  }
  if (d.stats_layout == THD_STATS_TOKEN_MAJOR) {
    p->stats_tok = d.h_q;
    p->stats_head = 1;
  } else {
    p->stats_tok = 1;
    p->stats_head = d.cap_rows_stats;
  }
  // non-overlapping O rows bound the number of (sequence, query tile) pairs
  const int64_t max_pairs = (int64_t)d.batch + (d.cap_rows[3] + p->rows_per_unit - 1) / p->rows_per_unit + 1;
  if (2 * max_pairs * d.h_q >= (int64_t(1) << 31)) {
    delete p;
    return THD_ERR_UNSUPPORTED;
  }
  p->max_pairs = (int32_t)max_pairs;
  // KV split (tensor-core path): it only triggers below kSplitWaves waves of units,
  // i.e. for fewer than kSplitWaves * SMs / h_q pairs, which bounds the split table
  // and the partial-result buffers
  p->allow_split = kernel == THD_KERNEL_TCGEN05 && !(d.flags & THD_FLAG_NO_KV_SPLIT);
  const int64_t split_bound = ((int64_t)thd::kSplitWaves * thd::kMaxSmsForSizing + d.h_q - 1) / d.h_q;
  p->max_split = p->allow_split ? (int32_t)(max_pairs < split_bound ? max_pairs : split_bound) : 0;
  p->max_tail = p->max_split < thd::max_tail_pairs(d.h_q) ? p->max_split : thd::max_tail_pairs(d.h_q);
  // partial slots: two per split pair, kTailParts per pair cut for the last wave;
  // the pair list holds every pair plus the extra parts of the split ones
  const int64_t slots = 2 * (int64_t)p->max_split + (int64_t)(thd::kTailParts - 2) * p->max_tail;
  const int64_t entries = max_pairs + (p->allow_split ? (int64_t)p->max_split + (thd::kTailParts - 2) * p->max_tail : 0);
  if (entries * d.h_q >= (int64_t(1) << 31)) {
    delete p;
    return THD_ERR_UNSUPPORTED;
  }
  p->pair_cap = (int32_t)entries;
  p->slot_cap = (int32_t)slots;
  const int64_t part_rows = slots * d.h_q * p->rows_per_unit;
  int64_t off = 0;
  p->ws_off[0] = off; off = align_up(off + thd::kHeaderBytes, kAlign);
  p->ws_off[1] = off; off = align_up(off + (int64_t)d.batch * (int64_t)sizeof(thd::SeqMeta), kAlign);
  p->ws_off[2] = off; off = align_up(off + ((int64_t)d.batch + 1) * 4, kAlign);
  p->ws_off[3] = off;
  off = align_up(off + entries * (int64_t)sizeof(thd::PairRec), kAlign);
  p->ws_off[4] = off; off = align_up(off + (int64_t)p->max_split * (int64_t)sizeof(thd::SplitRec), kAlign);
  p->ws_off[5] = off; off = align_up(off + part_rows * d.d * 4, kAlign);
  p->ws_off[6] = off; off = align_up(off + part_rows * 4, kAlign);
  p->ws_bytes = (size_t)off;
  *ws_bytes = p->ws_bytes;
  *out = p;
  return THD_OK;
}

thd_kernel_t thd_attn_plan_kernel(thd_attn_plan_t plan) { return plan ? plan->kernel : THD_KERNEL_AUTO; }

void thd_attn_plan_geometry(thd_attn_plan_t plan, int32_t* rows, int32_t* keys, int32_t* max_pairs) {
  if (!plan) return;
  if (rows) *rows = plan->rows_per_unit;
  if (keys) *keys = plan->keys_per_tile;
  if (max_pairs) *max_pairs = plan->max_pairs;
}

void thd_attn_plan_workspace_layout(thd_attn_plan_t plan, int64_t offsets[4]) {
  // the first four regions; the split table and partial buffers follow
  if (!plan || !offsets) return;
  for (int i = 0; i < 4; ++i) offsets[i] = plan->ws_off[i];
}

namespace {
void profile_release(thd_attn_plan_t plan) {
  if (plan->prof_events) {
    for (int i = 0; i < 2 * plan->prof_slots; ++i) cudaEventDestroy(plan->prof_events[i]);
    delete[] plan->prof_events;
  }
  plan->prof_events = nullptr;
  plan->prof_slots = 0;
  plan->prof_count = 0;
}
}  // namespace

void thd_attn_plan_destroy(thd_attn_plan_t plan) {
  if (!plan) return;
  profile_release(plan);
  delete plan;
}

thd_status_t thd_attn_profile_enable(thd_attn_plan_t plan, int32_t slots) {
  if (!plan || slots < 0) return THD_ERR_INVALID_ARG;
  profile_release(plan);
  if (slots == 0) return THD_OK;
  plan->prof_events = new (std::nothrow) cudaEvent_t[2 * slots];
  if (!plan->prof_events) return THD_ERR_INVALID_ARG;
  for (int i = 0; i < 2 * slots; ++i) {
    if (cudaEventCreate(&plan->prof_events[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(plan->prof_events[j]);
      delete[] plan->prof_events;
      plan->prof_events = nullptr;
      return THD_ERR_CUDA;
    }
  }
  plan->prof_slots = slots;
  plan->prof_count = 0;
  return THD_OK;
}

thd_status_t thd_attn_profile_read(thd_attn_plan_t plan, float* mean_ms, int32_t* launches) {
  if (!plan || !mean_ms || !launches) return THD_ERR_INVALID_ARG;
  double total = 0.0;
  const int n = plan->prof_count;
  for (int i = 0; i < n; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(plan->prof_events[2 * i + 1]) != cudaSuccess) return THD_ERR_CUDA;
    if (cudaEventElapsedTime(&ms, plan->prof_events[2 * i], plan->prof_events[2 * i + 1]) != cudaSuccess)
      return THD_ERR_CUDA;
    total += ms;
  }
  *mean_ms = n > 0 ? (float)(total / n) : 0.f;
  *launches = n;
  plan->prof_count = 0;
  return THD_OK;
}

thd_status_t thd_attn_fwd(thd_attn_plan_t plan, const void* q, const void* k, const void* v, void* o,
                          float* stats, const int32_t* cu_q, const int32_t* cu_k, const int32_t* off_q,
                          const int32_t* off_k, const int32_t* off_v, const int32_t* off_o,
                          const int32_t* off_s, const int8_t* mask, const int32_t* qco, void* workspace,
                          void* stream_ptr) {
  return thd_attn_fwd_window(plan, q, k, v, o, stats, cu_q, cu_k, off_q, off_k, off_v, off_o, off_s, mask, qco,
                             nullptr, workspace, stream_ptr);
}

thd_status_t thd_attn_fwd_window(thd_attn_plan_t plan, const void* q, const void* k, const void* v, void* o,
                                 float* stats, const int32_t* cu_q, const int32_t* cu_k, const int32_t* off_q,
                                 const int32_t* off_k, const int32_t* off_v, const int32_t* off_o,
                                 const int32_t* off_s, const int8_t* mask, const int32_t* qco,
                                 const int32_t* window_left, void* workspace, void* stream_ptr) {
  if (!plan || plan->is_bwd || plan->is_indexer) return THD_ERR_INVALID_ARG;
  const thd_attn_desc_t& d = plan->desc;
  if (!workspace) return THD_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return THD_ERR_WORKSPACE;
  // metadata is always read for every sequence; a tensor pointer may be NULL only
  // when its view has no rows (nothing can address it then)
  if (d.batch > 0 && (!cu_q || !cu_k || !off_q || !off_k || !off_v || !off_o || !off_s || !mask))
    return THD_ERR_INVALID_ARG;
  const void* tens[4] = {q, k, v, o};
  for (int i = 0; i < 4; ++i)
    if (!tens[i] && d.cap_rows[i] > 0) return THD_ERR_INVALID_ARG;
  if (!stats && d.cap_rows_stats > 0) return THD_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);

  thd::SetupParams sp;
  sp.cu_q = cu_q; sp.cu_k = cu_k;
  sp.off_q = off_q; sp.off_k = off_k; sp.off_v = off_v; sp.off_o = off_o; sp.off_s = off_s;
  sp.mask = mask; sp.qco = qco; sp.window = window_left;
  sp.cap_q = d.cap_rows[0]; sp.cap_k = d.cap_rows[1]; sp.cap_v = d.cap_rows[2]; sp.cap_o = d.cap_rows[3];
  sp.cap_s = d.cap_rows_stats;
  sp.batch = d.batch;
  sp.rows_per_unit = plan->rows_per_unit;
  sp.keys_per_tile = plan->keys_per_tile;
  sp.max_pairs = plan->max_pairs;
  sp.pair_cap = plan->pair_cap > 0 ? plan->pair_cap : plan->max_pairs;
  sp.slot_cap = plan->slot_cap;
  sp.h_q = d.h_q;
  sp.key_axis = 0;
  sp.max_len_k = 0;
  sp.unit_heads = d.h_q;
  sp.allow_split = plan->allow_split;
  sp.element_offsets = (d.flags & THD_FLAG_ELEMENT_OFFSETS) ? 1 : 0;
  sp.offset_multiplier = d.offset_multiplier > 0 ? d.offset_multiplier : 1;
  for (int i = 0; i < 4; ++i) sp.tok_stride[i] = d.stride_tok[i] > 0 ? d.stride_tok[i] : 1;
  sp.tok_stride[4] = plan->stats_tok > 0 ? plan->stats_tok : 1;
  sp.max_split = plan->max_split;
  sp.max_tail = plan->max_tail;
  sp.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]);
  sp.meta = reinterpret_cast<thd::SeqMeta*>(ws + plan->ws_off[1]);
  sp.pair_base = reinterpret_cast<int32_t*>(ws + plan->ws_off[2]);
  sp.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off[3]);
  sp.splits = reinterpret_cast<thd::SplitRec*>(ws + plan->ws_off[4]);

  thd::FwdParams fp;
  fp.q = q; fp.k = k; fp.v = v; fp.o = o; fp.stats = stats;
  for (int i = 0; i < 4; ++i) {
    fp.stride_tok[i] = d.stride_tok[i];
    fp.stride_head[i] = d.stride_head[i];
  }
  fp.stats_tok = plan->stats_tok;
  fp.stats_head = plan->stats_head;
  fp.h_q = d.h_q; fp.h_kv = d.h_kv; fp.d = d.d;
  fp.scale_log2 = plan->scale * 1.4426950408889634f;
  fp.header = sp.header;
  fp.counter = sp.header + thd::kHdrCounter;
  fp.status = sp.header + thd::kHdrStatus;
  fp.meta = sp.meta;
  fp.pairs = sp.pairs;
  fp.splits = sp.splits;
  fp.part_o = reinterpret_cast<float*>(ws + plan->ws_off[5]);
  fp.part_lse = reinterpret_cast<float*>(ws + plan->ws_off[6]);
  fp.rows_per_unit = plan->rows_per_unit;
  fp.test_stall = (d.flags & THD_FLAG_TEST_STALL) ? 1 : 0;
  fp.has_window = window_left != nullptr ? 1 : 0;

  // a view with no rows has no TMA descriptor: the SIMT kernel serves that call
  // (it walks any unit size, so the plan's schedule geometry still applies)
  bool use_tc = plan->kernel == THD_KERNEL_TCGEN05;
  for (int i = 0; i < 3; ++i)
    if (d.cap_rows[i] == 0) use_tc = false;
  if (use_tc) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if (a % 16 != 0) return THD_ERR_ALIGNMENT;
  }

  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return THD_ERR_CUDA;
  // the tensor-core kernel's persistent grid: one CTA per SM
  sp.num_ctas = use_tc ? thd::tc_grid_size(num_sms, plan->max_pairs, d.h_q) : num_sms;
  if (!use_tc) sp.allow_split = 0;
  if (thd::launch_setup(sp, stream) != cudaSuccess) return THD_ERR_CUDA;
  const bool prof = plan->prof_events && plan->prof_count < plan->prof_slots;
  if (prof && cudaEventRecord(plan->prof_events[2 * plan->prof_count], stream) != cudaSuccess)
    return THD_ERR_CUDA;
  cudaError_t err;
  if (use_tc) {
    err = thd::launch_fwd_tc(fp, d, plan->max_pairs, num_sms, stream);
    if (err == cudaErrorNotSupported) return THD_ERR_UNSUPPORTED;
    if (err == cudaSuccess && plan->allow_split) err = thd::launch_combine(fp, d.dtype, num_sms, stream);
  } else {
    err = thd::launch_fwd_simt(fp, d.dtype, plan->rows_per_unit, num_sms, stream);
  }
  if (err != cudaSuccess) return THD_ERR_CUDA;
  if (prof) {
    if (cudaEventRecord(plan->prof_events[2 * plan->prof_count + 1], stream) != cudaSuccess)
      return THD_ERR_CUDA;
    ++plan->prof_count;
  }
  return THD_OK;
}

thd_status_t thd_attn_read_status(thd_attn_plan_t plan, const void* workspace, uint32_t* host_out,
                                  void* stream_ptr) {
  if (!plan || !host_out) return THD_ERR_INVALID_ARG;
  if (!workspace) return THD_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const char* src = static_cast<const char*>(workspace) + plan->ws_off[0] + 4 * thd::kHdrStatus;
  uint32_t words[2] = {0u, 0u};
  if (cudaMemcpyAsync(&words[0], src, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return THD_ERR_CUDA;
  if (plan->is_bwd || indexer_uses_key_axis(plan)) {
    // the key-axis schedules of the backward and of the tensor-core indexer keep
    // their own status word
    const int64_t hdr = plan->is_bwd ? plan->ws_off_b[0] : plan->ws_off_b[1];
    const char* src_k = static_cast<const char*>(workspace) + hdr + 4 * thd::kHdrStatus;
    if (cudaMemcpyAsync(&words[1], src_k, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return THD_ERR_CUDA;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) return THD_ERR_CUDA;
  *host_out = words[0] | words[1];
  return THD_OK;
}

// ------------------------------------------------------------------------- backward

thd_status_t thd_attn_plan_bwd(thd_attn_plan_t* out, const thd_attn_bwd_desc_t* desc, size_t* ws_bytes) {
  if (!out || !desc || !ws_bytes) return THD_ERR_INVALID_ARG;
  *out = nullptr;
  const thd_attn_desc_t& d = desc->fwd;
  // the forward descriptor's own checks (views, capacities, scale, kernel request)
  thd_attn_plan_t fp = nullptr;
  size_t fws = 0;
  const thd_status_t st = thd_attn_plan(&fp, &d, &fws);
  if (st != THD_OK) return st;
  thd_attn_plan_destroy(fp);
  // gradient views: same dtype; each at least as many rows as its primal view
  // (dO <-> O, dQ <-> Q, dK <-> K, dV <-> V), and its all-axes span inside its bytes
  const int eb = elem_bytes(d.dtype);
  const int64_t prim_rows[4] = {d.cap_rows[3], d.cap_rows[0], d.cap_rows[1], d.cap_rows[2]};
  const int64_t heads[4] = {d.h_q, d.h_q, d.h_kv, d.h_kv};
  for (int i = 0; i < 4; ++i) {
    if (desc->cap_rows[i] < prim_rows[i] || desc->cap_rows[i] >= (int64_t(1) << 31)) return THD_ERR_INVALID_ARG;
    if (desc->stride_tok[i] < 0 || desc->stride_head[i] < 0 || desc->bytes[i] < 0) return THD_ERR_INVALID_ARG;
    if (desc->bytes[i] == 0) continue;
    const int64_t span = thd_attn_view_span_bytes(desc->cap_rows[i], heads[i], d.d, desc->stride_tok[i],
                                                  desc->stride_head[i], eb);
    if (span > desc->bytes[i]) return THD_ERR_CAPACITY;
  }
  // tensor-core backward: the forward's conditions, plus dO through TMA and 16-byte
  // gradient rows
  bool tc_ok = tc_applicable(d, scale_of(d));
  for (int i = 0; i < 4; ++i) {
    if (desc->stride_tok[i] <= 0 || desc->stride_head[i] <= 0) tc_ok = false;
    if ((desc->stride_tok[i] * eb) % 16 != 0 || (desc->stride_head[i] * eb) % 16 != 0) tc_ok = false;
  }
  thd_kernel_t kernel;
  if (d.kernel == THD_KERNEL_SIMT) {
    kernel = THD_KERNEL_SIMT;
  } else if (d.kernel == THD_KERNEL_TCGEN05) {
    if (!tc_ok) return THD_ERR_UNSUPPORTED;
    kernel = THD_KERNEL_TCGEN05;
  } else {
    kernel = tc_ok ? THD_KERNEL_TCGEN05 : THD_KERNEL_SIMT;
  }

  auto* p = new (std::nothrow) thd_attn_plan_s;
  if (!p) return THD_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->desc = d;
  p->is_bwd = 1;
  p->kernel = kernel;
  p->scale = scale_of(d);
  p->elem_bytes = eb;
  for (int i = 0; i < 4; ++i) {
    p->g_cap_rows[i] = desc->cap_rows[i];
    p->g_stride_tok[i] = desc->stride_tok[i];
    p->g_stride_head[i] = desc->stride_head[i];
  }
  p->rows_per_unit = thd::kBwdRowsPerUnit;
  p->keys_per_tile = thd::kBwdKeysPerUnit;
  if (d.stats_layout == THD_STATS_TOKEN_MAJOR) {
    p->stats_tok = d.h_q;
    p->stats_head = 1;
  } else {
    p->stats_tok = 1;
    p->stats_head = d.cap_rows_stats;
  }
  // non-overlapping Q rows bound the query-axis pairs, non-overlapping K rows the key-axis ones
  const int64_t max_q = (int64_t)d.batch + (d.cap_rows[0] + p->rows_per_unit - 1) / p->rows_per_unit + 1;
  const int64_t max_k = (int64_t)d.batch + (d.cap_rows[1] + thd::kBwdKeysPerUnit - 1) / thd::kBwdKeysPerUnit + 1;
  if (max_q * d.h_q >= (int64_t(1) << 31) || max_k * d.h_kv >= (int64_t(1) << 31)) {
    delete p;
    return THD_ERR_UNSUPPORTED;
  }
  p->max_pairs = (int32_t)max_q;
  p->max_pairs_k = (int32_t)max_k;
  p->allow_split = 0;
  p->max_split = 0;
  p->max_tail = 0;
  int64_t off = 0;
  p->ws_off[0] = off; off = align_up(off + thd::kHeaderBytes, kAlign);
  p->ws_off[1] = off; off = align_up(off + (int64_t)d.batch * (int64_t)sizeof(thd::SeqMeta), kAlign);
  p->ws_off[2] = off; off = align_up(off + ((int64_t)d.batch + 1) * 4, kAlign);
  p->ws_off[3] = off; off = align_up(off + max_q * (int64_t)sizeof(thd::PairRec), kAlign);
  p->ws_off[4] = p->ws_off[5] = p->ws_off[6] = off;
  p->ws_off_b[0] = off; off = align_up(off + thd::kHeaderBytes, kAlign);
  p->ws_off_b[1] = off; off = align_up(off + ((int64_t)d.batch + 1) * 4, kAlign);
  p->ws_off_b[2] = off; off = align_up(off + max_k * (int64_t)sizeof(thd::PairRec), kAlign);
  p->ws_off_b[3] = off; off = align_up(off + max_q * d.h_q * thd::kBwdRowsPerUnit * 8, kAlign);
  p->ws_bytes = (size_t)off;
  *ws_bytes = p->ws_bytes;
  *out = p;
  return THD_OK;
}

thd_status_t thd_attn_bwd(thd_attn_plan_t plan, const void* q, const void* k, const void* v, const void* o,
                          const void* d_o, const float* stats, void* dq, void* dk, void* dv, const int32_t* cu_q,
                          const int32_t* cu_k, const int32_t* off_q, const int32_t* off_k, const int32_t* off_v,
                          const int32_t* off_o, const int32_t* off_s, const int8_t* mask, const int32_t* qco,
                          const int32_t* window_left, void* workspace, void* stream_ptr) {
  if (!plan || !plan->is_bwd) return THD_ERR_INVALID_ARG;
  const thd_attn_desc_t& d = plan->desc;
  if (!workspace) return THD_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return THD_ERR_WORKSPACE;
  if (d.batch > 0 && (!cu_q || !cu_k || !off_q || !off_k || !off_v || !off_o || !off_s || !mask))
    return THD_ERR_INVALID_ARG;
  const void* prim[4] = {q, k, v, o};
  for (int i = 0; i < 4; ++i)
    if (!prim[i] && d.cap_rows[i] > 0) return THD_ERR_INVALID_ARG;
  const void* grads[4] = {d_o, dq, dk, dv};
  for (int i = 0; i < 4; ++i)
    if (!grads[i] && plan->g_cap_rows[i] > 0) return THD_ERR_INVALID_ARG;
  if (!stats && d.cap_rows_stats > 0) return THD_ERR_INVALID_ARG;
  // every check that can fail comes before the first launch
  // a view with no rows has no TMA descriptor: the SIMT kernels serve that call
  bool use_tc = plan->kernel == THD_KERNEL_TCGEN05;
  for (int i = 0; i < 3; ++i)
    if (d.cap_rows[i] == 0) use_tc = false;
  if (plan->g_cap_rows[0] == 0) use_tc = false;
  if (use_tc) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(d_o) |
                        reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
                        reinterpret_cast<uintptr_t>(dv);
    if (a % 16 != 0) return THD_ERR_ALIGNMENT;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return THD_ERR_CUDA;

  thd::SetupParams sp;
  sp.cu_q = cu_q; sp.cu_k = cu_k;
  sp.off_q = off_q; sp.off_k = off_k; sp.off_v = off_v; sp.off_o = off_o; sp.off_s = off_s;
  sp.mask = mask; sp.qco = qco; sp.window = window_left;
  sp.cap_q = d.cap_rows[0]; sp.cap_k = d.cap_rows[1]; sp.cap_v = d.cap_rows[2]; sp.cap_o = d.cap_rows[3];
  sp.cap_s = d.cap_rows_stats;
  sp.batch = d.batch;
  sp.h_q = d.h_q;
  sp.max_len_k = 0;
  sp.allow_split = 0;
  sp.element_offsets = (d.flags & THD_FLAG_ELEMENT_OFFSETS) ? 1 : 0;
  sp.offset_multiplier = d.offset_multiplier > 0 ? d.offset_multiplier : 1;
  for (int i = 0; i < 4; ++i) sp.tok_stride[i] = d.stride_tok[i] > 0 ? d.stride_tok[i] : 1;
  sp.tok_stride[4] = plan->stats_tok > 0 ? plan->stats_tok : 1;
  sp.max_split = 0;
  sp.max_tail = 0;
  sp.num_ctas = num_sms;
  sp.meta = reinterpret_cast<thd::SeqMeta*>(ws + plan->ws_off[1]);
  sp.splits = nullptr;
  // query axis: dQ units of rows_per_unit rows, cost in KV tiles
  sp.key_axis = 0;
  sp.unit_heads = d.h_q;
  sp.rows_per_unit = plan->rows_per_unit;
  sp.keys_per_tile = thd::kBwdKeysPerUnit;
  sp.max_pairs = plan->max_pairs;
  sp.pair_cap = plan->pair_cap > 0 ? plan->pair_cap : plan->max_pairs;
  sp.slot_cap = plan->slot_cap;
  sp.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]);
  sp.pair_base = reinterpret_cast<int32_t*>(ws + plan->ws_off[2]);
  sp.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off[3]);
  if (thd::launch_setup(sp, stream) != cudaSuccess) return THD_ERR_CUDA;
  thd::BwdParams bp;
  bp.header_q = sp.header;
  bp.counter_q = sp.header + thd::kHdrCounter;
  bp.pairs_q = sp.pairs;
  // key axis: dK/dV units of kBwdKeysPerUnit keys, cost in query tiles
  sp.key_axis = 1;
  sp.group_keys = 1;
  sp.unit_heads = d.h_kv;
  sp.rows_per_unit = thd::kBwdKeysPerUnit;
  sp.keys_per_tile = plan->rows_per_unit;
  sp.max_pairs = plan->max_pairs_k;
  sp.pair_cap = plan->max_pairs_k;
  sp.slot_cap = 0;
  sp.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off_b[0]);
  sp.pair_base = reinterpret_cast<int32_t*>(ws + plan->ws_off_b[1]);
  sp.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off_b[2]);
  if (thd::launch_setup(sp, stream) != cudaSuccess) return THD_ERR_CUDA;
  bp.header_k = sp.header;
  bp.counter_k = sp.header + thd::kHdrCounter;
  bp.pairs_k = sp.pairs;

  bp.q = q; bp.k = k; bp.v = v; bp.o = o; bp.d_o = d_o; bp.stats = stats;
  bp.dq = dq; bp.dk = dk; bp.dv = dv;
  for (int i = 0; i < 4; ++i) {
    bp.stride_tok[i] = d.stride_tok[i];
    bp.stride_head[i] = d.stride_head[i];
    bp.stride_tok[4 + i] = plan->g_stride_tok[i];
    bp.stride_head[4 + i] = plan->g_stride_head[i];
  }
  bp.stats_tok = plan->stats_tok;
  bp.stats_head = plan->stats_head;
  bp.h_q = d.h_q; bp.h_kv = d.h_kv; bp.d = d.d;
  bp.scale = plan->scale;
  bp.scale_log2 = plan->scale * 1.4426950408889634f;
  bp.status = const_cast<uint32_t*>(bp.header_q) + thd::kHdrStatus;
  bp.meta = sp.meta;
  bp.ld = reinterpret_cast<float2*>(ws + plan->ws_off_b[3]);
  bp.pair_base_q = reinterpret_cast<const int32_t*>(ws + plan->ws_off[2]);
  bp.rows_per_unit = plan->rows_per_unit;
  bp.keys_per_unit = thd::kBwdKeysPerUnit;
  bp.has_window = window_left != nullptr ? 1 : 0;

  if (thd::launch_bwd_prep(bp, d.dtype, num_sms, stream) != cudaSuccess) return THD_ERR_CUDA;
  const bool prof = plan->prof_events && plan->prof_count < plan->prof_slots;
  if (prof && cudaEventRecord(plan->prof_events[2 * plan->prof_count], stream) != cudaSuccess)
    return THD_ERR_CUDA;
  if (use_tc) {
    const cudaError_t err = thd::launch_bwd_tc(bp, d, plan->g_cap_rows, plan->g_stride_tok, plan->g_stride_head,
                                               plan->max_pairs, plan->max_pairs_k, num_sms, stream);
    if (err == cudaErrorNotSupported) return THD_ERR_UNSUPPORTED;
    if (err != cudaSuccess) return THD_ERR_CUDA;
  } else if (thd::launch_bwd_simt(bp, d.dtype, num_sms, stream) != cudaSuccess) {
    return THD_ERR_CUDA;
  }
  if (prof) {
    if (cudaEventRecord(plan->prof_events[2 * plan->prof_count + 1], stream) != cudaSuccess)
      return THD_ERR_CUDA;
    ++plan->prof_count;
  }
  return THD_OK;
}

// -------------------------------------------------------------------------- indexer

thd_status_t thd_indexer_plan(thd_attn_plan_t* out, const thd_indexer_desc_t* desc, size_t* ws_bytes) {
  if (!out || !desc || !ws_bytes) return THD_ERR_INVALID_ARG;
  *out = nullptr;
  const thd_indexer_desc_t& d = *desc;
  if (d.dtype != THD_BF16 && d.dtype != THD_FP16) return THD_ERR_INVALID_ARG;
  if (d.batch < 0 || d.heads < 1 || d.heads > 128 || d.d < 1 || d.d > 128) return THD_ERR_INVALID_ARG;
  if (d.topk < 1 || d.topk > thd::kIndexerMaxTopk) return THD_ERR_INVALID_ARG;
  if (d.flags != 0) return THD_ERR_INVALID_ARG;
  if (d.kernel != THD_KERNEL_AUTO && d.kernel != THD_KERNEL_SIMT && d.kernel != THD_KERNEL_TCGEN05)
    return THD_ERR_INVALID_ARG;
  const int64_t caps[3] = {d.cap_rows_q, d.cap_rows_k, d.cap_rows_out};
  for (int i = 0; i < 3; ++i)
    if (caps[i] < 0 || caps[i] >= (int64_t(1) << 31)) return THD_ERR_INVALID_ARG;
  if (d.stride_tok_q < 0 || d.stride_head_q < 0 || d.stride_tok_k < 0 || d.stride_tok_w < 0 || d.max_seqlen_k < 0)
    return THD_ERR_INVALID_ARG;
  const bool tc_ok = thd::indexer_tc_applicable(d);
  if (d.kernel == THD_KERNEL_TCGEN05 && !tc_ok) return THD_ERR_UNSUPPORTED;
  auto* p = new (std::nothrow) thd_attn_plan_s;
  if (!p) return THD_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->is_indexer = 1;
  p->idesc = d;
  p->kernel = (d.kernel != THD_KERNEL_SIMT && tc_ok) ? THD_KERNEL_TCGEN05 : THD_KERNEL_SIMT;
  p->elem_bytes = 2;
  p->rows_per_unit = thd::kIndexerRowsPerUnit;
  p->keys_per_tile = 128;
  const int64_t max_len = d.max_seqlen_k > 0 ? d.max_seqlen_k : d.cap_rows_k;
  p->score_row = align_up(max_len > 0 ? max_len : 1, 128);
  const int64_t max_pairs = (int64_t)d.batch + (d.cap_rows_out + p->rows_per_unit - 1) / p->rows_per_unit + 1;
  p->max_pairs = (int32_t)max_pairs;
  // key-axis units (tensor-core scores): sequences may share key rows (the query
  // chunks of one document under context parallelism all read its key prefix), so
  // the bound is per sequence: len_k <= max_len (checked on the device)
  const int64_t max_k =
      (int64_t)d.batch * ((max_len + thd::kIndexerKeysPerUnit - 1) / thd::kIndexerKeysPerUnit) + 1;
  if (max_k >= (int64_t(1) << 31) || max_pairs >= (int64_t(1) << 31)) {
    delete p;
    return THD_ERR_UNSUPPORTED;
  }
  p->max_pairs_k = (int32_t)max_k;
  int64_t off = 0;
  p->ws_off[0] = off; off = align_up(off + thd::kHeaderBytes, kAlign);
  p->ws_off[1] = off; off = align_up(off + (int64_t)d.batch * (int64_t)sizeof(thd::SeqMeta), kAlign);
  p->ws_off[2] = off; off = align_up(off + ((int64_t)d.batch + 1) * 4, kAlign);
  p->ws_off[3] = off; off = align_up(off + max_pairs * (int64_t)sizeof(thd::PairRec), kAlign);
  p->ws_off[4] = p->ws_off[5] = p->ws_off[6] = off;
  p->ws_off_b[0] = off; off = align_up(off + d.cap_rows_out * p->score_row * 4, kAlign);
  p->ws_off_b[1] = off; off = align_up(off + thd::kHeaderBytes, kAlign);
  p->ws_off_b[2] = off; off = align_up(off + ((int64_t)d.batch + 1) * 4, kAlign);
  p->ws_off_b[3] = off; off = align_up(off + max_k * (int64_t)sizeof(thd::PairRec), kAlign);
  p->ws_bytes = (size_t)off;
  *ws_bytes = p->ws_bytes;
  *out = p;
  return THD_OK;
}

thd_status_t thd_indexer_topk(thd_attn_plan_t plan, const void* q_i, const void* k_i, const float* w,
                              int32_t* idx_out, float* score_out, const int32_t* cu_q, const int32_t* cu_k,
                              const int32_t* off_q, const int32_t* off_k, const int32_t* off_out, const int8_t* mask,
                              const int32_t* qco, void* workspace, void* stream_ptr) {
  if (!plan || !plan->is_indexer) return THD_ERR_INVALID_ARG;
  const thd_indexer_desc_t& d = plan->idesc;
  if (!workspace) return THD_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return THD_ERR_WORKSPACE;
  if (d.batch > 0 && (!cu_q || !cu_k || !off_q || !off_k || !off_out || !mask)) return THD_ERR_INVALID_ARG;
  if ((!q_i || !w) && d.cap_rows_q > 0) return THD_ERR_INVALID_ARG;
  if (!k_i && d.cap_rows_k > 0) return THD_ERR_INVALID_ARG;
  if (!idx_out && d.cap_rows_out > 0) return THD_ERR_INVALID_ARG;
  // every check that can fail comes before the first launch, so that a status read
  // after a successful call always sees headers this call's setup kernels wrote
  const bool use_tc = indexer_uses_key_axis(plan);
  if (use_tc) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(q_i) | reinterpret_cast<uintptr_t>(k_i) |
                        reinterpret_cast<uintptr_t>(w);
    if (a % 16 != 0) return THD_ERR_ALIGNMENT;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  char* ws = static_cast<char*>(workspace);
  const int num_sms = num_sms_of_current_device();
  if (num_sms <= 0) return THD_ERR_CUDA;
  thd::SetupParams sp;
  sp.cu_q = cu_q; sp.cu_k = cu_k;
  sp.off_q = off_q; sp.off_k = off_k; sp.off_v = off_k; sp.off_o = off_out; sp.off_s = off_out;
  sp.mask = mask; sp.qco = qco; sp.window = nullptr;
  sp.cap_q = d.cap_rows_q; sp.cap_k = d.cap_rows_k; sp.cap_v = d.cap_rows_k; sp.cap_o = d.cap_rows_out;
  sp.cap_s = d.cap_rows_out;
  sp.batch = d.batch;
  sp.rows_per_unit = plan->rows_per_unit;
  sp.keys_per_tile = plan->keys_per_tile;
  sp.max_pairs = plan->max_pairs;
  sp.pair_cap = plan->pair_cap > 0 ? plan->pair_cap : plan->max_pairs;
  sp.slot_cap = plan->slot_cap;
  sp.h_q = 1;
  sp.key_axis = 0;
  sp.max_len_k = d.max_seqlen_k;   // 0: len_k <= cap_rows_k <= the score row already
  sp.unit_heads = 1;
  sp.allow_split = 0;
  sp.element_offsets = 0;
  sp.offset_multiplier = 1;
  for (int i = 0; i < 5; ++i) sp.tok_stride[i] = 1;
  sp.num_ctas = num_sms;
  sp.max_split = 0;
  sp.max_tail = 0;
  sp.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]);
  sp.meta = reinterpret_cast<thd::SeqMeta*>(ws + plan->ws_off[1]);
  sp.pair_base = reinterpret_cast<int32_t*>(ws + plan->ws_off[2]);
  sp.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off[3]);
  sp.splits = nullptr;
  if (thd::launch_setup(sp, stream) != cudaSuccess) return THD_ERR_CUDA;
  thd::IndexerParams ip;
  ip.header_k = nullptr;
  ip.counter_k = nullptr;
  ip.pairs_k = nullptr;
  if (use_tc) {
    // key-axis schedule for the tensor-core scores (units of 256 keys)
    sp.key_axis = 1;
    sp.rows_per_unit = thd::kIndexerKeysPerUnit;
    sp.keys_per_tile = 128;
    sp.max_pairs = plan->max_pairs_k;
    sp.pair_cap = plan->max_pairs_k;
    sp.slot_cap = 0;
    sp.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off_b[1]);
    sp.pair_base = reinterpret_cast<int32_t*>(ws + plan->ws_off_b[2]);
    sp.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off_b[3]);
    if (thd::launch_setup(sp, stream) != cudaSuccess) return THD_ERR_CUDA;
    ip.header_k = sp.header;
    ip.counter_k = sp.header + thd::kHdrCounter;
    ip.pairs_k = sp.pairs;
  }
  ip.q = q_i; ip.k = k_i; ip.w = w; ip.idx = idx_out; ip.score_out = score_out;
  ip.scores = reinterpret_cast<float*>(ws + plan->ws_off_b[0]);
  ip.q_tok = d.stride_tok_q; ip.q_head = d.stride_head_q; ip.k_tok = d.stride_tok_k; ip.w_tok = d.stride_tok_w;
  ip.score_row = plan->score_row;
  ip.heads = d.heads; ip.d = d.d; ip.topk = d.topk;
  ip.header = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]);
  ip.counter = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]) + thd::kHdrCounter;
  ip.pairs = reinterpret_cast<thd::PairRec*>(ws + plan->ws_off[3]);
  ip.meta = sp.meta;
  ip.status = reinterpret_cast<uint32_t*>(ws + plan->ws_off[0]) + thd::kHdrStatus;
  const bool prof = plan->prof_events && plan->prof_count < plan->prof_slots;
  if (prof && cudaEventRecord(plan->prof_events[2 * plan->prof_count], stream) != cudaSuccess)
    return THD_ERR_CUDA;
  if (use_tc) {
    const cudaError_t err = thd::launch_indexer_scores_tc(ip, d, plan->max_pairs_k, num_sms, stream);
    if (err == cudaErrorNotSupported) return THD_ERR_UNSUPPORTED;
    if (err != cudaSuccess) return THD_ERR_CUDA;
  } else if (thd::launch_indexer_scores_simt(ip, d.dtype, num_sms, stream) != cudaSuccess) {
    return THD_ERR_CUDA;
  }
  if (prof) {
    if (cudaEventRecord(plan->prof_events[2 * plan->prof_count + 1], stream) != cudaSuccess) return THD_ERR_CUDA;
    ++plan->prof_count;
  }
  if (thd::launch_indexer_topk(ip, num_sms, stream) != cudaSuccess) return THD_ERR_CUDA;
  return THD_OK;
}

}  // extern "C"
