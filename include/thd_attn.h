/*
 * thd_attn.h -- C ABI of the GB300 (sm_103a) packed-THD attention library
 * (forward; its backward and the sparse-attention indexer top-k at the end of
 * this file).
 *
 * Operation (scaled-dot-product attention forward with log-sum-exp Stats over a
 * packed, ragged "THD" batch):
 *
 *   for each sequence b and query head h (kv head g = h / (h_q / h_kv)):
 *     len_q = cu_seqlens_q[b+1] - cu_seqlens_q[b],  len_k = cu_seqlens_kv[b+1] - cu_seqlens_kv[b]
 *     q_i = Q[off_q[b] + i, h, :],  k_j = K[off_k[b] + j, g, :],  v_j = V[off_v[b] + j, g, :]
 *     s_ij = softmax_scale * <q_i, k_j>
 *     visible(i, j) = j < len_k  and  (mask 0: true | mask 1: j <= i | mask 2: j <= i + c)
 *         c = q_causal_offset[b], or len_k - len_q when q_causal_offset is NULL
 *     LSE_i = ln sum_{visible j} exp(s_ij)               (natural log, scaled scores)
 *     O_i   = sum_{visible j} exp(s_ij - LSE_i) * v_j
 *     rows with no visible key: O_i = 0, LSE_i = -inf
 *     O[off_o[b] + i, h, :] = O_i ;  Stats[(off_s[b] + i) * st_tok + h * st_head] = LSE_i
 *
 *   Every other row of O and Stats is left untouched (pad rows are never written).
 *
 * Where each piece comes from:
 *   - per-tensor ragged offsets, read on the device instead of re-deriving
 *     prefix(lens) x stride; lengths still drive the mask bounds and dead rows:
 *     cuDNN-frontend issue "THD lowering never reads the bound ragged offsets",
 *     sections "Concrete failure" and "Proposal: consume the bound offsets on device";
 *   - cu_seqlens / cu_seqlens_padded vocabulary, per-sequence mask policy as an
 *     on-device tensor, no host synchronisation in the call:
 *     TransformerEngine PR #3274, review comments on pad_between_seqs and
 *     attn_mask_type_per_seq;
 *   - q_causal_offset ("global token index of each segment's local q[0]") and
 *     bottom-right alignment for context-parallel chunks: Megatron-LM PR #14
 *     "fix(dsa): align packed-CP indexer causal masks";
 *   - Stats layouts token-major [t,h] and head-major [h,t], the all-axes span rule
 *     for capacities, and the persistent scheduler's tile counter at word 0 of the
 *     workspace: NVIDIA/cudnn-frontend PR #462, sections "What", "Root cause" and
 *     "The fix".
 *   - 16-byte alignment of pointers and token strides: cudnn-frontend PR #516
 *     (ragged token-stride gaps), squashed commit text.
 *
 * Conventions:
 *   - All tensors are caller-owned device memory. The library allocates no device
 *     memory in thd_attn_fwd; scratch lives in the caller's workspace.
 *   - Offsets are ROW units per tensor; element address of (row, head, e) in Q/K/V/O
 *     is base + row * stride_tok + head * stride_head + e (elements; last dim contiguous).
 *   - Host-side errors are returned as thd_status_t; nothing aborts or throws.
 *   - Device-side data errors (bad lengths/offsets/mask values) are recorded as bits
 *     in a status word inside the workspace; the affected sequence gets no work and
 *     its rows stay untouched. thd_attn_read_status copies that word to the host.
 *   - thd_attn_fwd is asynchronous on the given stream, performs no device->host
 *     read and no allocation, and may be captured in a CUDA graph.
 */
#ifndef THD_ATTN_H
#define THD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  THD_OK = 0,
  THD_ERR_INVALID_ARG = 1,   /* bad descriptor field or NULL pointer */
  THD_ERR_UNSUPPORTED = 2,   /* valid request the selected kernel cannot serve */
  THD_ERR_ALIGNMENT = 3,     /* pointer or stride not 16-byte aligned where required */
  THD_ERR_CAPACITY = 4,      /* a tensor view's all-axes span exceeds its declared bytes */
  THD_ERR_WORKSPACE = 5,     /* workspace NULL, too small, or misaligned */
  THD_ERR_CUDA = 6           /* a CUDA runtime call or kernel launch failed */
} thd_status_t;

typedef enum { THD_BF16 = 0, THD_FP16 = 1, THD_FP32 = 2 } thd_dtype_t;

/* Stats (LSE) layout: token-major [t, h] (token stride h_q, head stride 1) or
 * head-major [h, t] (token stride 1, head stride cap_rows_stats). */
typedef enum { THD_STATS_TOKEN_MAJOR = 0, THD_STATS_HEAD_MAJOR = 1 } thd_stats_layout_t;

/* Kernel choice. AUTO takes the tcgen05 tensor-core kernel where it applies
 * (bf16/fp16, d in {64, 128}, 16-byte aligned rows) and the SIMT kernel
 * otherwise; the other two force one (TCGEN05 fails with THD_ERR_UNSUPPORTED
 * when it does not apply). */
typedef enum { THD_KERNEL_AUTO = 0, THD_KERNEL_SIMT = 1, THD_KERNEL_TCGEN05 = 2 } thd_kernel_t;

/* Mask policy values of the per-sequence mask_type tensor. */
enum { THD_MASK_NONE = 0, THD_MASK_CAUSAL_TOP_LEFT = 1, THD_MASK_CAUSAL_BOTTOM_RIGHT = 2 };

/* Bits of the device status word (thd_attn_read_status). */
enum {
  THD_DEV_BAD_LENGTH = 1u << 0,     /* cu_seqlens not non-decreasing for some b */
  THD_DEV_BAD_OFFSET = 1u << 1,     /* off[b] < 0 or off[b] + len > cap_rows for some tensor */
  THD_DEV_BAD_MASK = 1u << 2,       /* mask_type[b] not in {0, 1, 2} */
  THD_DEV_TILE_OVERFLOW = 1u << 3,  /* more work units than the plan's capacity (no work done) */
  THD_DEV_WAIT_TIMEOUT = 1u << 4,   /* a bounded in-kernel wait gave up (kernel returned early) */
  THD_DEV_KEY_OVERLAP = 1u << 5     /* backward: K or V rows of two sequences overlap without the
                                       sequences forming one key group (see thd_attn_bwd); no dK
                                       or dV row is written */
};

/* Host-known problem description, fixed per plan. Index 0..3 of the stride and
 * capacity arrays is Q, K, V, O. */
typedef struct {
  thd_dtype_t dtype;              /* storage type of Q, K, V and O */
  int32_t batch;                  /* B, number of sequences (>= 0) */
  int32_t h_q, h_kv, d;           /* heads and head dim; h_q % h_kv == 0; 1 <= d <= 128 */
  int64_t cap_rows[4];            /* physical rows of the Q, K, V, O views */
  int64_t stride_tok[4];          /* elements between consecutive rows */
  int64_t stride_head[4];         /* elements between consecutive heads */
  int64_t bytes[4];               /* allocation size behind each pointer (bytes); the view's
                                     all-axes span must fit. 0 = not checked */
  int64_t cap_rows_stats;         /* physical rows of Stats (T_s) */
  thd_stats_layout_t stats_layout;
  float softmax_scale;            /* NaN => 1/sqrt(d) */
  thd_kernel_t kernel;
  uint32_t flags;                 /* THD_FLAG_* bits */
  int32_t offset_multiplier;      /* with THD_FLAG_ELEMENT_OFFSETS: factor applied on the device
                                     to every offset (0 or 1: none) */
} thd_attn_desc_t;

/* Plan flags.
 * THD_FLAG_NO_KV_SPLIT: never split a unit's key range. By default, when a launch
 *   has fewer than about four waves of work units for the GPU, the tensor-core
 *   path processes long units as two halves of their key range (and the cheapest
 *   long ones whose units would make up a last, partial wave as eight parts) and
 *   merges the parts' partial results (log-sum-exp weighted) in a small follow-up
 *   kernel, which evens out the end of the launch. The partial results live in the
 *   workspace, so splitting enlarges workspace_bytes; this flag keeps it small. */
enum { THD_FLAG_NO_KV_SPLIT = 1u << 0 };
/* THD_FLAG_ELEMENT_OFFSETS: the five offset arrays hold ELEMENT offsets, the
 * convention where a sequence's offset is its first row times the tensor's token
 * stride (Stats: times the Stats token stride), optionally scaled by
 * offset_multiplier (applied on the device, like a ragged-offset multiplier).
 * The setup kernel divides each by the tensor's token stride; an offset that is
 * not a whole number of rows sets THD_DEV_BAD_OFFSET and that sequence gets no
 * work (cuDNN-frontend issue "THD lowering never reads the bound ragged offsets",
 * the element-vs-byte convention and multiplier notes; NVIDIA/cudnn-frontend PR
 * #462, "Not addressed here": ragged_offset == cum_token x stride[2]). */
enum { THD_FLAG_ELEMENT_OFFSETS = 1u << 1 };
/* THD_FLAG_TEST_STALL: test hook for the bounded-wait path of the tensor-core
 * kernel. The MMA-issuing thread waits on a barrier that nothing completes, gives
 * up after 100 ms, sets THD_DEV_WAIT_TIMEOUT in the status word, and every CTA
 * drains and returns. Outputs are undefined after such a call; the CUDA context
 * stays usable. Never set it outside tests. */
enum { THD_FLAG_TEST_STALL = 1u << 31 };

typedef struct thd_attn_plan_s* thd_attn_plan_t;

/* Validate the descriptor and pick the kernel (host only: no CUDA call, no device
 * read). On success *out owns a plan (free with thd_attn_plan_destroy) and
 * *workspace_bytes is the scratch the fwd call needs (256-byte aligned device
 * memory; its first word is the persistent scheduler's tile counter). */
thd_status_t thd_attn_plan(thd_attn_plan_t* out, const thd_attn_desc_t* desc,
                           size_t* workspace_bytes);

/* Enqueue the forward pass on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   q, k, v, o        device pointers to the views described by the plan
 *   stats             device float32 LSE buffer (layout per plan)
 *   cu_seqlens_q/kv   device int32 [B+1]; per-sequence lengths are the differences
 *   off_q .. off_s    device int32 [>= B] row offset of each sequence's first row in
 *                     Q, K, V, O and Stats (a cu_seqlens_padded array may be passed
 *                     directly; entry B is not read)
 *   mask_type         device int8 [B], values THD_MASK_*
 *   q_causal_offset   device int32 [B] or NULL (NULL => len_k - len_q for mask 2;
 *                     ignored for masks 0 and 1)
 *   workspace         device memory of >= workspace_bytes, 256-byte aligned
 * Returns THD_OK once both kernels are enqueued. Device data errors surface only
 * through thd_attn_read_status. Sequences whose O (or Stats) rows overlap race. */
thd_status_t thd_attn_fwd(thd_attn_plan_t plan, const void* q, const void* k, const void* v,
                          void* o, float* stats, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_kv, const int32_t* off_q,
                          const int32_t* off_k, const int32_t* off_v, const int32_t* off_o,
                          const int32_t* off_s, const int8_t* mask_type,
                          const int32_t* q_causal_offset, void* workspace, void* stream);

/* thd_attn_fwd with a per-sequence left window on the causal masks.
 *   window_left   device int32 [B] or NULL. For a sequence with mask 1 or 2 and
 *                 window_left[b] = w >= 0, row i sees keys i + c - w .. i + c
 *                 (c = 0 for mask 1; bounded causal attention); w < 0, mask 0 or
 *                 NULL leave the lower end unbounded. TransformerEngine PR #3274
 *                 describes per-policy windows for such bounded causal attention.
 * All other arguments and results as in thd_attn_fwd, which equals this call with
 * window_left = NULL. */
thd_status_t thd_attn_fwd_window(thd_attn_plan_t plan, const void* q, const void* k, const void* v,
                                 void* o, float* stats, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_kv, const int32_t* off_q,
                                 const int32_t* off_k, const int32_t* off_v, const int32_t* off_o,
                                 const int32_t* off_s, const int8_t* mask_type,
                                 const int32_t* q_causal_offset, const int32_t* window_left,
                                 void* workspace, void* stream);

/* Copy the device status word of the last call on this workspace (fwd, bwd or
 * indexer top-k with this plan; the OR of both schedules' words where a call
 * builds two) to *host_out and synchronise `stream`. This is the only call that
 * waits on the device. */
thd_status_t thd_attn_read_status(thd_attn_plan_t plan, const void* workspace,
                                  uint32_t* host_out, void* stream);

/* Which kernel the plan selected: THD_KERNEL_SIMT or THD_KERNEL_TCGEN05. */
thd_kernel_t thd_attn_plan_kernel(thd_attn_plan_t plan);

/* Tile geometry the plan uses (query rows per scheduled unit, keys per KV tile)
 * and its capacity in scheduled (sequence, query-tile) pairs. */
void thd_attn_plan_geometry(thd_attn_plan_t plan, int32_t* rows_per_unit,
                            int32_t* keys_per_tile, int32_t* max_pairs);

/* Byte offsets, inside the workspace, of its first four regions: [0] header words
 * (tile counter, status, entry count, tile count, first entry of each cost group,
 * split count), [1] per-sequence metadata (12 int32 per sequence: len_q, len_k,
 * off_q, off_k, off_v, off_o, off_s, shift, window lower shift, 3 unused), [2]
 * per-sequence first pair index
 * (int32 [B+1]), [3] the scheduled entry list (int32 {b, first query row,
 * (part << 8) | parts, partial slot or -1} per entry, longest first). For
 * inspection only. */
void thd_attn_plan_workspace_layout(thd_attn_plan_t plan, int64_t offsets[4]);

void thd_attn_plan_destroy(thd_attn_plan_t plan);

/* Kernel timing for benchmarks. After thd_attn_profile_enable(plan, slots > 0),
 * each thd_attn_fwd on this plan records a CUDA event pair around the attention
 * kernel alone (not the setup kernel) on its stream, for up to `slots` calls.
 * thd_attn_profile_read waits for the recorded events, returns the mean
 * attention-kernel time in milliseconds and the number of launches it covers,
 * and starts a new recording. slots = 0 turns recording off. Not for use while
 * a stream is being captured into a CUDA graph. */
thd_status_t thd_attn_profile_enable(thd_attn_plan_t plan, int32_t slots);
thd_status_t thd_attn_profile_read(thd_attn_plan_t plan, float* mean_ms, int32_t* launches);

const char* thd_attn_status_string(thd_status_t status);

/* All-axes span in bytes of a strided view: ((rows-1)*s_t + (heads-1)*s_h + (d-1) + 1) * elem,
 * 0 for an empty view (the workspace-sizing rule of cudnn-frontend PR #462, "The fix"). */
int64_t thd_attn_view_span_bytes(int64_t rows, int64_t heads, int64_t d, int64_t stride_tok,
                                 int64_t stride_head, int64_t elem_bytes);

/* Forward pass without a caller workspace, for callers that cannot allocate
 * device memory where they run attention (inside a stream being captured into
 * a CUDA graph, in plugins whose host runtime owns all device memory, or in
 * serving loops that cannot afford an allocator's implicit synchronisation).
 * No counterpart exists in the pages this library follows; it is an addition
 * for such callers.
 *
 * Same arguments and results as thd_attn_fwd minus `workspace`. The scratch is a
 * static device array of thd_attn_static_workspace_capacity() bytes (1 MiB) that
 * each GPU loading this library keeps until the process exits. The call makes no
 * allocation of any kind. Returns THD_ERR_INVALID_ARG for a backward or indexer
 * plan, and THD_ERR_WORKSPACE when a forward plan's workspace_bytes exceed that
 * capacity (plan with THD_FLAG_NO_KV_SPLIT: the partial results of split key
 * ranges do not fit the static array).
 *
 * The first call on each device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress; make it before any stream capture.
 * All calls on a device share the array, which keeps the previous call's
 * contents (each call rewrites what it reads before reading it). Calls that
 * overlap on the GPU -- e.g. on unordered streams -- race on the array. The
 * device status word of these calls lives in that array: read it with
 * thd_attn_static_read_status. */
thd_status_t thd_attn_fwd_static_ws(thd_attn_plan_t plan, const void* q, const void* k, const void* v,
                                    void* o, float* stats, const int32_t* cu_seqlens_q,
                                    const int32_t* cu_seqlens_kv, const int32_t* off_q,
                                    const int32_t* off_k, const int32_t* off_v, const int32_t* off_o,
                                    const int32_t* off_s, const int8_t* mask_type,
                                    const int32_t* q_causal_offset, void* stream);

/* Capacity in bytes of the static scratch array used by thd_attn_fwd_static_ws. */
size_t thd_attn_static_workspace_capacity(void);

/* thd_attn_read_status for calls made through thd_attn_fwd_static_ws: copies the
 * device status word that the last such call on the current device left in the
 * static array (THD_DEV_* bits) to *host_out and synchronises `stream`. `plan`
 * must be the forward plan of that call. Like thd_attn_fwd_static_ws it has no
 * counterpart in the pages; it waits on the device, so it is not for use while a
 * stream is being captured. */
thd_status_t thd_attn_static_read_status(thd_attn_plan_t plan, uint32_t* host_out, void* stream);

/* ------------------------------------------------------------------ backward
 *
 * Gradients of the forward pass above (ragged SDPA backward over the same
 * metadata and Stats layouts: NVIDIA/cudnn-frontend PR #462, sections "What" and
 * "Root cause", which name the backward's per-row softmax sums and dQ/dK/dV
 * intermediates in THD layout). For an upstream gradient dO (the loss is
 * L = sum_i <O_i, dO_i>), per sequence b and query head h (kv head g):
 *
 *     P_ij  = exp(s_ij - LSE_i) on visible keys, 0 elsewhere (LSE_i read from Stats)
 *     D_i   = <dO_i, O_i>                               (O read from the O view)
 *     dV_j  = sum_i P_ij dO_i
 *     dS_ij = P_ij (<dO_i, v_j> - D_i)
 *     dQ_i  = softmax_scale * sum_j dS_ij k_j
 *     dK_j  = softmax_scale * sum_i dS_ij q_i
 *
 *   dK and dV of kv head g sum over the query heads of its group. dQ rows are
 *   written at off_q[b] + i, dK rows at off_k[b] + j, dV rows at off_v[b] + j
 *   (each gradient shares its primal tensor's row offsets); dO is read at
 *   off_o[b] + i. A query row with no visible key gets dQ = 0; a key no query
 *   sees gets dK = dV = 0. Rows outside the sequences are never written.
 *   Masks, causal offsets and windows as in thd_attn_fwd_window.
 */
typedef struct {
  thd_attn_desc_t fwd;            /* the forward's Q, K, V, O views, Stats, scale, kernel, flags */
  int64_t cap_rows[4];            /* index 0..3: dO, dQ, dK, dV views (same dtype as the forward); */
  int64_t stride_tok[4];          /*   each gradient view needs at least its primal view's rows */
  int64_t stride_head[4];
  int64_t bytes[4];               /* 0 = not checked */
} thd_attn_bwd_desc_t;

/* Validate a backward descriptor and pick the kernels (host only). The plan is
 * used with thd_attn_bwd (not thd_attn_fwd); *workspace_bytes as for thd_attn_plan.
 * THD_FLAG_ELEMENT_OFFSETS and THD_FLAG_NO_KV_SPLIT are accepted; element offsets
 * of dO / dQ / dK / dV follow their primal tensors' token strides. */
thd_status_t thd_attn_plan_bwd(thd_attn_plan_t* out, const thd_attn_bwd_desc_t* desc,
                               size_t* workspace_bytes);

/* Enqueue the backward pass on `stream`.
 *   q, k, v, o, stats  the forward's inputs, output and LSE (read only)
 *   d_o                upstream gradient, dO view of the plan (read only)
 *   dq, dk, dv         gradient views of the plan (written rows only)
 *   remaining metadata as in thd_attn_fwd_window (window_left may be NULL)
 * Asynchronous, no allocation, no device->host read; device data errors surface
 * through thd_attn_read_status.
 *
 * Sequences may share key rows: consecutive sequences whose off_k AND off_v are
 * equal form one key group (e.g. the zigzag query chunks of one document under
 * context parallelism, each bottom-right at its own q_causal_offset over a prefix
 * of the document's keys; Megatron-LM PR #14). Each dK / dV row of a group is the
 * sum over all of its members that see the key, and is written once. K or V rows
 * shared in any other way (partial overlaps, equal offsets that are not adjacent
 * in the batch) set THD_DEV_KEY_OVERLAP and no dK / dV row is written. dQ rows of
 * different sequences that overlap race. */
thd_status_t thd_attn_bwd(thd_attn_plan_t plan, const void* q, const void* k, const void* v,
                          const void* o, const void* d_o, const float* stats, void* dq, void* dk,
                          void* dv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                          const int32_t* off_q, const int32_t* off_k, const int32_t* off_v,
                          const int32_t* off_o, const int32_t* off_s, const int8_t* mask_type,
                          const int32_t* q_causal_offset, const int32_t* window_left,
                          void* workspace, void* stream);

/* ------------------------------------------------------------ indexer top-k
 *
 * Sparse-attention indexer over a packed THD batch: per query row, score every
 * visible key and keep the top-k (Megatron-LM PR #14 "fix(dsa): align packed-CP
 * indexer causal masks": the indexer masks each THD segment with the same causal
 * policy as attention, bottom-right with q_causal_offset for context-parallel
 * chunks, then selects the best keys per row). The pages do not print the score;
 * this library computes the lightning-indexer score of DeepSeek-V3.2 sparse
 * attention, with H indexer heads:
 *
 *     I_ij = sum_h  w_ih * max(0, <q_ih, k_j>)       (fp32 accumulation)
 *
 *   q_i = QI[off_q[b] + i, h, :], k_j = KI[off_k[b] + j, :] (one indexer key per
 *   token), w_ih = W[off_q[b] + i, h] (float32; any scale folded in). Visible keys
 *   as in thd_attn_fwd (mask 0 / 1 / 2, q_causal_offset). For each row, idx_out
 *   row off_out[b] + i receives the sequence-local numbers j of the min(topk,
 *   visible) visible keys of largest I_ij, ordered by descending score (equal
 *   scores: ascending j), then -1; score_out (optional) the matching scores, NaN
 *   in unused slots. Rows outside the sequences are never written.
 */
typedef struct {
  thd_dtype_t dtype;              /* QI and KI storage: THD_BF16 or THD_FP16 */
  int32_t batch;
  int32_t heads;                  /* H, 1..128 */
  int32_t d;                      /* 1..128 */
  int32_t topk;                   /* 1..2048 */
  int64_t cap_rows_q, stride_tok_q, stride_head_q;  /* QI view [rows, H, d]; W has the same rows */
  int64_t cap_rows_k, stride_tok_k;                  /* KI view [rows, d] */
  int64_t stride_tok_w;           /* float32 W [cap_rows_q, H], head stride 1 */
  int64_t cap_rows_out;           /* idx_out int32 [rows, topk] and score_out float32 [rows, topk] */
  int64_t max_seqlen_k;           /* bound on len_k for the score scratch (0 = cap_rows_k); a
                                     longer sequence sets THD_DEV_BAD_LENGTH and gets no work */
  thd_kernel_t kernel;
  uint32_t flags;                 /* none defined; must be 0 */
} thd_indexer_desc_t;

/* Validate and size (host only). The workspace holds the schedules and a float32
 * score row of max_seqlen_k entries (rounded up to 128) per output row. Segments
 * may share key rows (the zigzag query chunks of one document under context
 * parallelism all read its key prefix): the key-axis schedule is sized per
 * segment from max_seqlen_k, not from cap_rows_k. */
thd_status_t thd_indexer_plan(thd_attn_plan_t* out, const thd_indexer_desc_t* desc, size_t* workspace_bytes);

/* Enqueue the indexer top-k (asynchronous, no allocation, no device->host read).
 * score_out may be NULL. Offsets are row offsets into QI (and W), KI and the
 * outputs; off_out[b] addresses both idx_out and score_out. */
thd_status_t thd_indexer_topk(thd_attn_plan_t plan, const void* q_i, const void* k_i, const float* w,
                              int32_t* idx_out, float* score_out, const int32_t* cu_seqlens_q,
                              const int32_t* cu_seqlens_kv, const int32_t* off_q, const int32_t* off_k,
                              const int32_t* off_out, const int8_t* mask_type,
                              const int32_t* q_causal_offset, void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* THD_ATTN_H */
