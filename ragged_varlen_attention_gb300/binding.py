"""ctypes binding of ``libthd_attn.so`` (declared in ``include/thd_attn.h``).

Argument marshalling only: torch tensors become device pointers, strides and
sizes; every step of the forward pass runs in the library's CUDA kernels. There
is no fallback -- when the library is missing the first call raises.
"""
from __future__ import annotations

import collections
import ctypes
import math
import os

import torch

STATS_TOKEN_MAJOR, STATS_HEAD_MAJOR = 0, 1
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TCGEN05 = 0, 1, 2
FLAG_NO_KV_SPLIT = 1
FLAG_ELEMENT_OFFSETS = 2
FLAG_TEST_STALL = 1 << 31
_DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
_STATUS = {0: "THD_OK", 1: "THD_ERR_INVALID_ARG", 2: "THD_ERR_UNSUPPORTED",
           3: "THD_ERR_ALIGNMENT", 4: "THD_ERR_CAPACITY", 5: "THD_ERR_WORKSPACE",
           6: "THD_ERR_CUDA"}

# device status word bits
DEV_BAD_LENGTH, DEV_BAD_OFFSET, DEV_BAD_MASK, DEV_TILE_OVERFLOW, DEV_WAIT_TIMEOUT = 1, 2, 4, 8, 16
DEV_KEY_OVERLAP = 32


class ThdAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}")
        self.status = status


class ThdAttnDesc(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("batch", ctypes.c_int32),
        ("h_q", ctypes.c_int32),
        ("h_kv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("cap_rows", ctypes.c_int64 * 4),
        ("stride_tok", ctypes.c_int64 * 4),
        ("stride_head", ctypes.c_int64 * 4),
        ("bytes", ctypes.c_int64 * 4),
        ("cap_rows_stats", ctypes.c_int64),
        ("stats_layout", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("kernel", ctypes.c_int),
        ("flags", ctypes.c_uint32),
        ("offset_multiplier", ctypes.c_int32),
    ]


class ThdAttnBwdDesc(ctypes.Structure):
    _fields_ = [
        ("fwd", ThdAttnDesc),
        ("cap_rows", ctypes.c_int64 * 4),      # dO, dQ, dK, dV
        ("stride_tok", ctypes.c_int64 * 4),
        ("stride_head", ctypes.c_int64 * 4),
        ("bytes", ctypes.c_int64 * 4),
    ]


class ThdIndexerDesc(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("batch", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("cap_rows_q", ctypes.c_int64),
        ("stride_tok_q", ctypes.c_int64),
        ("stride_head_q", ctypes.c_int64),
        ("cap_rows_k", ctypes.c_int64),
        ("stride_tok_k", ctypes.c_int64),
        ("stride_tok_w", ctypes.c_int64),
        ("cap_rows_out", ctypes.c_int64),
        ("max_seqlen_k", ctypes.c_int64),
        ("kernel", ctypes.c_int),
        ("flags", ctypes.c_uint32),
    ]


_LIB = None
_EXPORTS = ["thd_attn_plan", "thd_attn_fwd", "thd_attn_read_status", "thd_attn_plan_kernel",
            "thd_attn_plan_geometry", "thd_attn_plan_workspace_layout", "thd_attn_plan_destroy",
            "thd_attn_status_string", "thd_attn_view_span_bytes", "thd_attn_profile_enable",
            "thd_attn_profile_read", "thd_attn_fwd_static_ws", "thd_attn_static_workspace_capacity",
            "thd_attn_static_read_status",
            "thd_attn_fwd_window", "thd_attn_plan_bwd", "thd_attn_bwd", "thd_indexer_plan",
            "thd_indexer_topk"]


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libthd_attn.so")


def load_library():
    """Load the C-ABI library once; raise if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with ragged_varlen_attention_gb300.build")
    lib = ctypes.CDLL(path)
    vp, i32p, i64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    lib.thd_attn_plan.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(ThdAttnDesc),
                                  ctypes.POINTER(ctypes.c_size_t)]
    lib.thd_attn_plan.restype = ctypes.c_int
    lib.thd_attn_fwd.argtypes = [vp] * 17
    lib.thd_attn_fwd.restype = ctypes.c_int
    lib.thd_attn_fwd_window.argtypes = [vp] * 18
    lib.thd_attn_fwd_window.restype = ctypes.c_int
    lib.thd_attn_plan_bwd.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(ThdAttnBwdDesc),
                                      ctypes.POINTER(ctypes.c_size_t)]
    lib.thd_attn_plan_bwd.restype = ctypes.c_int
    lib.thd_attn_bwd.argtypes = [vp] * 22
    lib.thd_attn_bwd.restype = ctypes.c_int
    lib.thd_indexer_plan.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(ThdIndexerDesc),
                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.thd_indexer_plan.restype = ctypes.c_int
    lib.thd_indexer_topk.argtypes = [vp] * 15
    lib.thd_indexer_topk.restype = ctypes.c_int
    lib.thd_attn_read_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.thd_attn_read_status.restype = ctypes.c_int
    lib.thd_attn_plan_kernel.argtypes = [vp]
    lib.thd_attn_plan_kernel.restype = ctypes.c_int
    lib.thd_attn_plan_geometry.argtypes = [vp, i32p, i32p, i32p]
    lib.thd_attn_plan_geometry.restype = None
    lib.thd_attn_plan_workspace_layout.argtypes = [vp, i64p]
    lib.thd_attn_plan_workspace_layout.restype = None
    lib.thd_attn_plan_destroy.argtypes = [vp]
    lib.thd_attn_plan_destroy.restype = None
    lib.thd_attn_status_string.argtypes = [ctypes.c_int]
    lib.thd_attn_status_string.restype = ctypes.c_char_p
    lib.thd_attn_view_span_bytes.argtypes = [ctypes.c_int64] * 6
    lib.thd_attn_view_span_bytes.restype = ctypes.c_int64
    lib.thd_attn_profile_enable.argtypes = [vp, ctypes.c_int32]
    lib.thd_attn_profile_enable.restype = ctypes.c_int
    lib.thd_attn_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i32p]
    lib.thd_attn_profile_read.restype = ctypes.c_int
    lib.thd_attn_fwd_static_ws.argtypes = [vp] * 16
    lib.thd_attn_fwd_static_ws.restype = ctypes.c_int
    lib.thd_attn_static_workspace_capacity.argtypes = []
    lib.thd_attn_static_workspace_capacity.restype = ctypes.c_size_t
    lib.thd_attn_static_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.thd_attn_static_read_status.restype = ctypes.c_int
    _LIB = lib
    return lib


class ThdAttnPlan:
    """Owns a ``thd_attn_plan_t`` (forward, backward or indexer plan); frees it when
    collected."""

    def __init__(self, handle: int, workspace_bytes: int, desc: ThdAttnDesc):
        self.handle = handle
        self.workspace_bytes = workspace_bytes
        self.desc = desc
        lib = load_library()
        self.kernel = lib.thd_attn_plan_kernel(handle)
        a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        lib.thd_attn_plan_geometry(handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        self.rows_per_unit, self.keys_per_tile, self.max_pairs = a.value, b.value, c.value
        offs = (ctypes.c_int64 * 4)()
        lib.thd_attn_plan_workspace_layout(handle, offs)
        self.workspace_layout = tuple(int(x) for x in offs)

    def __del__(self):
        if getattr(self, "handle", None) and _LIB is not None:
            _LIB.thd_attn_plan_destroy(self.handle)
            self.handle = None


def _view_bytes(t: torch.Tensor) -> int:
    return t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()


def make_desc(dtype: torch.dtype, batch: int, h_q: int, h_kv: int, d: int, cap_rows, stride_tok,
              stride_head, nbytes=(0, 0, 0, 0), cap_rows_stats: int = 0,
              stats_layout: int = STATS_TOKEN_MAJOR, softmax_scale: float | None = None,
              kernel: int = KERNEL_AUTO, flags: int = 0, offset_multiplier: int = 0) -> ThdAttnDesc:
    desc = ThdAttnDesc()
    desc.dtype = _DTYPE_CODE[dtype]
    desc.batch, desc.h_q, desc.h_kv, desc.d = batch, h_q, h_kv, d
    for i in range(4):
        desc.cap_rows[i] = int(cap_rows[i])
        desc.stride_tok[i] = int(stride_tok[i])
        desc.stride_head[i] = int(stride_head[i])
        desc.bytes[i] = int(nbytes[i])
    desc.cap_rows_stats = int(cap_rows_stats)
    desc.stats_layout = int(stats_layout)
    desc.softmax_scale = math.nan if softmax_scale is None else float(softmax_scale)
    desc.kernel = int(kernel)
    desc.flags = int(flags)
    desc.offset_multiplier = int(offset_multiplier)
    return desc


def thd_attn_plan(desc: ThdAttnDesc) -> ThdAttnPlan:
    lib = load_library()
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_attn_plan(ctypes.byref(handle), ctypes.byref(desc), ctypes.byref(ws))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_plan")
    return ThdAttnPlan(handle.value, ws.value, desc)


def plan_for_tensors(q, k, v, o, batch: int, cap_rows_stats: int, stats_layout: int,
                     softmax_scale=None, kernel: int = KERNEL_AUTO, flags: int = 0,
                     offset_multiplier: int = 0) -> ThdAttnPlan:
    """Build a plan from [rows, heads, d] tensor views (last dim contiguous)."""
    for t in (q, k, v, o):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("Q/K/V/O must be [rows, heads, d] views with a contiguous last dim")
        if t.dtype != q.dtype:
            raise ValueError("Q, K, V and O must share one storage type")
    desc = make_desc(q.dtype, batch, q.shape[1], k.shape[1], q.shape[2],
                     [t.shape[0] for t in (q, k, v, o)], [t.stride(0) for t in (q, k, v, o)],
                     [t.stride(1) for t in (q, k, v, o)], [_view_bytes(t) for t in (q, k, v, o)],
                     cap_rows_stats, stats_layout, softmax_scale, kernel, flags, offset_multiplier)
    return thd_attn_plan(desc)


def plan_bwd_for_tensors(q, k, v, o, d_o, dq, dk, dv, batch: int, cap_rows_stats: int,
                         stats_layout: int, softmax_scale=None, kernel: int = KERNEL_AUTO,
                         flags: int = 0, offset_multiplier: int = 0) -> ThdAttnPlan:
    """Backward plan from [rows, heads, d] views of the forward's tensors and of the
    gradients dO, dQ, dK, dV (see ``thd_attn_plan_bwd`` in include/thd_attn.h)."""
    for t in (q, k, v, o, d_o, dq, dk, dv):
        if t.dim() != 3 or t.stride(2) != 1:
            raise ValueError("tensors must be [rows, heads, d] views with a contiguous last dim")
        if t.dtype != q.dtype:
            raise ValueError("the forward's tensors and the gradients must share one storage type")
    bd = ThdAttnBwdDesc()
    bd.fwd = make_desc(q.dtype, batch, q.shape[1], k.shape[1], q.shape[2],
                       [t.shape[0] for t in (q, k, v, o)], [t.stride(0) for t in (q, k, v, o)],
                       [t.stride(1) for t in (q, k, v, o)], [_view_bytes(t) for t in (q, k, v, o)],
                       cap_rows_stats, stats_layout, softmax_scale, kernel, flags, offset_multiplier)
    for i, t in enumerate((d_o, dq, dk, dv)):
        bd.cap_rows[i] = t.shape[0]
        bd.stride_tok[i] = t.stride(0)
        bd.stride_head[i] = t.stride(1)
        bd.bytes[i] = _view_bytes(t)
    lib = load_library()
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_attn_plan_bwd(ctypes.byref(handle), ctypes.byref(bd), ctypes.byref(ws))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_plan_bwd")
    return ThdAttnPlan(handle.value, ws.value, bd.fwd)


def indexer_plan_for_tensors(q_i, k_i, w, idx_out, batch: int, topk: int, max_seqlen_k: int = 0,
                             kernel: int = KERNEL_AUTO) -> ThdAttnPlan:
    """Indexer plan from QI [rows, H, d], KI [rows, d], W [rows, H] (float32, head
    stride 1) and the int32 [rows, topk] output (see ``thd_indexer_plan``)."""
    if q_i.dim() != 3 or q_i.stride(2) != 1 or k_i.dim() != 2 or k_i.stride(1) != 1:
        raise ValueError("QI must be [rows, H, d] and KI [rows, d] with a contiguous last dim")
    if k_i.dtype != q_i.dtype:
        raise ValueError("QI and KI must share one storage type")
    if w.dtype != torch.float32 or w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("W must be float32 [rows, H] with head stride 1")
    if idx_out.dtype != torch.int32 or idx_out.dim() != 2 or idx_out.shape[1] != topk or not idx_out.is_contiguous():
        raise ValueError("idx_out must be a contiguous int32 [rows, topk] tensor")
    d = ThdIndexerDesc()
    d.dtype = _DTYPE_CODE[q_i.dtype]
    d.batch, d.heads, d.d, d.topk = batch, q_i.shape[1], q_i.shape[2], topk
    d.cap_rows_q, d.stride_tok_q, d.stride_head_q = q_i.shape[0], q_i.stride(0), q_i.stride(1)
    d.cap_rows_k, d.stride_tok_k = k_i.shape[0], k_i.stride(0)
    d.stride_tok_w = w.stride(0)
    d.cap_rows_out = idx_out.shape[0]
    d.max_seqlen_k = int(max_seqlen_k)
    d.kernel = int(kernel)
    d.flags = 0
    lib = load_library()
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = lib.thd_indexer_plan(ctypes.byref(handle), ctypes.byref(d), ctypes.byref(ws))
    if st != 0:
        raise ThdAttnError(st, "thd_indexer_plan")
    return ThdAttnPlan(handle.value, ws.value, d)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def thd_attn_fwd(plan: ThdAttnPlan, q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv, off_q, off_k,
                 off_v, off_o, off_s, mask_type, q_causal_offset, workspace, stream=None) -> None:
    """Enqueue the forward pass (see ``thd_attn_fwd`` in include/thd_attn.h)."""
    lib = load_library()
    st = lib.thd_attn_fwd(ctypes.c_void_p(plan.handle), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                          _ptr(stats), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(off_q),
                          _ptr(off_k), _ptr(off_v), _ptr(off_o), _ptr(off_s), _ptr(mask_type),
                          _ptr(q_causal_offset), _ptr(workspace), _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_fwd")


def thd_attn_fwd_window(plan: ThdAttnPlan, q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv, off_q,
                        off_k, off_v, off_o, off_s, mask_type, q_causal_offset, window_left,
                        workspace, stream=None) -> None:
    """Enqueue the forward pass with a per-sequence left window on the causal masks
    (see ``thd_attn_fwd_window`` in include/thd_attn.h); ``window_left`` is a device
    int32 [B] tensor or None."""
    lib = load_library()
    st = lib.thd_attn_fwd_window(ctypes.c_void_p(plan.handle), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                 _ptr(stats), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(off_q),
                                 _ptr(off_k), _ptr(off_v), _ptr(off_o), _ptr(off_s), _ptr(mask_type),
                                 _ptr(q_causal_offset), _ptr(window_left), _ptr(workspace),
                                 _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_fwd_window")


def thd_attn_bwd(plan: ThdAttnPlan, q, k, v, o, d_o, stats, dq, dk, dv, cu_seqlens_q,
                 cu_seqlens_kv, off_q, off_k, off_v, off_o, off_s, mask_type, q_causal_offset,
                 window_left, workspace, stream=None) -> None:
    """Enqueue the backward pass (see ``thd_attn_bwd`` in include/thd_attn.h)."""
    lib = load_library()
    st = lib.thd_attn_bwd(ctypes.c_void_p(plan.handle), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o),
                          _ptr(stats), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q),
                          _ptr(cu_seqlens_kv), _ptr(off_q), _ptr(off_k), _ptr(off_v), _ptr(off_o),
                          _ptr(off_s), _ptr(mask_type), _ptr(q_causal_offset), _ptr(window_left),
                          _ptr(workspace), _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_bwd")


def thd_indexer_topk(plan: ThdAttnPlan, q_i, k_i, w, idx_out, score_out, cu_seqlens_q, cu_seqlens_kv,
                     off_q, off_k, off_out, mask_type, q_causal_offset, workspace, stream=None) -> None:
    """Enqueue the indexer top-k (see ``thd_indexer_topk`` in include/thd_attn.h)."""
    lib = load_library()
    st = lib.thd_indexer_topk(ctypes.c_void_p(plan.handle), _ptr(q_i), _ptr(k_i), _ptr(w), _ptr(idx_out),
                              _ptr(score_out), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(off_q),
                              _ptr(off_k), _ptr(off_out), _ptr(mask_type), _ptr(q_causal_offset),
                              _ptr(workspace), _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_indexer_topk")


def thd_attn_fwd_static_ws(plan: ThdAttnPlan, q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv, off_q,
                           off_k, off_v, off_o, off_s, mask_type, q_causal_offset, stream=None) -> None:
    """Enqueue the forward pass with the library's static scratch array instead of a
    caller workspace (see ``thd_attn_fwd_static_ws`` in include/thd_attn.h): for
    callers that cannot allocate device memory where they run attention."""
    lib = load_library()
    st = lib.thd_attn_fwd_static_ws(ctypes.c_void_p(plan.handle), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(stats), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), _ptr(off_q),
                                    _ptr(off_k), _ptr(off_v), _ptr(off_o), _ptr(off_s), _ptr(mask_type),
                                    _ptr(q_causal_offset), _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_fwd_static_ws")


def static_workspace_capacity() -> int:
    return int(load_library().thd_attn_static_workspace_capacity())


def thd_attn_static_read_status(plan: ThdAttnPlan, stream=None) -> int:
    """Device status word (THD_DEV_* bits) of the last ``thd_attn_fwd_static_ws`` call
    on the current device; synchronises ``stream``."""
    out = ctypes.c_uint32()
    st = load_library().thd_attn_static_read_status(ctypes.c_void_p(plan.handle), ctypes.byref(out),
                                                     _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_static_read_status")
    return out.value


def thd_attn_read_status(plan: ThdAttnPlan, workspace, stream=None) -> int:
    lib = load_library()
    out = ctypes.c_uint32()
    st = lib.thd_attn_read_status(ctypes.c_void_p(plan.handle), _ptr(workspace), ctypes.byref(out),
                                  _stream_handle(stream))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_read_status")
    return out.value


def profile_enable(plan: ThdAttnPlan, slots: int) -> None:
    """Record CUDA events around the attention kernel of the next ``slots`` fwd calls."""
    st = load_library().thd_attn_profile_enable(ctypes.c_void_p(plan.handle), int(slots))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_profile_enable")


def profile_read(plan: ThdAttnPlan) -> tuple[float, int]:
    """(mean attention-kernel ms, launches recorded) since ``profile_enable``."""
    ms, n = ctypes.c_float(), ctypes.c_int32()
    st = load_library().thd_attn_profile_read(ctypes.c_void_p(plan.handle), ctypes.byref(ms),
                                              ctypes.byref(n))
    if st != 0:
        raise ThdAttnError(st, "thd_attn_profile_read")
    return float(ms.value), int(n.value)


def alloc_workspace(plan: ThdAttnPlan, device) -> torch.Tensor:
    n = max(256, (plan.workspace_bytes + 255) // 256 * 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


# plans of the one-call wrappers, keyed by everything a plan depends on; bounded
# (least recently used first out) so that a caller whose shapes keep changing does
# not accumulate plans: an evicted plan is destroyed once nothing references it
_PLAN_CACHE_SIZE = 64
_PLAN_CACHE: "collections.OrderedDict[tuple, ThdAttnPlan]" = collections.OrderedDict()


def _cached_plan(key: tuple, make):
    plan = _PLAN_CACHE.get(key)
    if plan is None:
        plan = make()
        _PLAN_CACHE[key] = plan
        while len(_PLAN_CACHE) > _PLAN_CACHE_SIZE:
            _PLAN_CACHE.popitem(last=False)
    else:
        _PLAN_CACHE.move_to_end(key)
    return plan


def thd_attn_forward(q, k, v, cu_seqlens_q, cu_seqlens_kv, *, off_q=None, off_k=None, off_v=None,
                     off_o=None, off_s=None, mask_type=None, q_causal_offset=None, o=None,
                     stats=None, stats_layout: int = STATS_TOKEN_MAJOR, softmax_scale=None,
                     kernel: int = KERNEL_AUTO, workspace=None, stream=None, window_left=None):
    """One-call forward over device tensors.

    Offsets default to the cu_seqlens arrays (packed layout); ``mask_type``
    defaults to no mask. O and Stats are allocated when not given (O with the
    shape of Q; Stats with Q's rows). ``window_left`` (device int32 [B]) bounds
    the causal masks from the left. Returns ``(o, stats)``.
    """
    batch = cu_seqlens_q.numel() - 1
    dev = q.device
    off_q = cu_seqlens_q if off_q is None else off_q
    off_k = cu_seqlens_kv if off_k is None else off_k
    off_v = off_k if off_v is None else off_v
    off_o = off_q if off_o is None else off_o
    off_s = off_o if off_s is None else off_s
    if mask_type is None:
        mask_type = torch.zeros(max(batch, 1), dtype=torch.int8, device=dev)
    if o is None:
        o = torch.zeros(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=dev)
    if stats is None:
        stats = torch.full((q.shape[0] * q.shape[1],), float("-inf"), dtype=torch.float32, device=dev)
    cap_s = stats.numel() // q.shape[1]
    key = (q.dtype, batch, tuple(q.shape), tuple(k.shape), tuple(v.shape), tuple(o.shape),
           q.stride(), k.stride(), v.stride(), o.stride(), cap_s, stats_layout, softmax_scale, kernel,
           _view_bytes(q), _view_bytes(k), _view_bytes(v), _view_bytes(o))
    plan = _cached_plan(key, lambda: plan_for_tensors(q, k, v, o, batch, cap_s, stats_layout, softmax_scale,
                                                      kernel))
    if workspace is None:
        workspace = alloc_workspace(plan, dev)
    thd_attn_fwd_window(plan, q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_v,
                        off_o, off_s, mask_type, q_causal_offset, window_left, workspace, stream)
    return o, stats


def thd_attn_backward(q, k, v, o, d_o, stats, cu_seqlens_q, cu_seqlens_kv, *, off_q=None, off_k=None,
                      off_v=None, off_o=None, off_s=None, mask_type=None, q_causal_offset=None,
                      window_left=None, dq=None, dk=None, dv=None, stats_layout: int = STATS_TOKEN_MAJOR,
                      softmax_scale=None, kernel: int = KERNEL_AUTO, workspace=None, stream=None):
    """One-call backward over device tensors (``thd_attn_bwd``): the gradients of
    the forward whose O and Stats are given, for the upstream gradient ``d_o``.
    Offsets and masks default as in :func:`thd_attn_forward`; gradients are
    allocated zero-filled when not given. Returns ``(dq, dk, dv)``."""
    batch = cu_seqlens_q.numel() - 1
    dev = q.device
    off_q = cu_seqlens_q if off_q is None else off_q
    off_k = cu_seqlens_kv if off_k is None else off_k
    off_v = off_k if off_v is None else off_v
    off_o = off_q if off_o is None else off_o
    off_s = off_o if off_s is None else off_s
    if mask_type is None:
        mask_type = torch.zeros(max(batch, 1), dtype=torch.int8, device=dev)
    dq = torch.zeros_like(q) if dq is None else dq
    dk = torch.zeros_like(k) if dk is None else dk
    dv = torch.zeros_like(v) if dv is None else dv
    cap_s = stats.numel() // q.shape[1]
    key = ("bwd", q.dtype, batch, tuple(q.shape), tuple(k.shape), tuple(v.shape), tuple(o.shape),
           q.stride(), k.stride(), v.stride(), o.stride(), d_o.stride(), dq.stride(), dk.stride(), dv.stride(),
           tuple(d_o.shape), tuple(dq.shape), tuple(dk.shape), tuple(dv.shape), cap_s, stats_layout,
           softmax_scale, kernel)
    plan = _cached_plan(key, lambda: plan_bwd_for_tensors(q, k, v, o, d_o, dq, dk, dv, batch, cap_s, stats_layout,
                                                          softmax_scale, kernel))
    if workspace is None:
        workspace = alloc_workspace(plan, dev)
    thd_attn_bwd(plan, q, k, v, o, d_o, stats, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_v,
                 off_o, off_s, mask_type, q_causal_offset, window_left, workspace, stream)
    return dq, dk, dv


def thd_indexer(q_i, k_i, w, cu_seqlens_q, cu_seqlens_kv, topk: int, *, off_q=None, off_k=None,
                off_out=None, mask_type=None, q_causal_offset=None, max_seqlen_k: int = 0,
                idx_out=None, score_out=None, with_scores: bool = True, kernel: int = KERNEL_AUTO,
                workspace=None, stream=None):
    """One-call indexer top-k (``thd_indexer_topk``) over device tensors: QI
    [rows, H, d], KI [rows, d], W float32 [rows, H]. Outputs have QI's rows unless
    given. Returns ``(idx int32 [rows, topk], scores float32 [rows, topk] or None)``."""
    batch = cu_seqlens_q.numel() - 1
    dev = q_i.device
    off_q = cu_seqlens_q if off_q is None else off_q
    off_k = cu_seqlens_kv if off_k is None else off_k
    off_out = off_q if off_out is None else off_out
    if mask_type is None:
        mask_type = torch.zeros(max(batch, 1), dtype=torch.int8, device=dev)
    if idx_out is None:
        idx_out = torch.full((q_i.shape[0], topk), -1, dtype=torch.int32, device=dev)
    if score_out is None and with_scores:
        score_out = torch.full((idx_out.shape[0], topk), float("nan"), dtype=torch.float32, device=dev)
    key = ("indexer", q_i.dtype, batch, tuple(q_i.shape), q_i.stride(), tuple(k_i.shape), k_i.stride(),
           w.stride(), tuple(idx_out.shape), topk, max_seqlen_k, kernel)
    plan = _cached_plan(key, lambda: indexer_plan_for_tensors(q_i, k_i, w, idx_out, batch, topk, max_seqlen_k,
                                                              kernel))
    if workspace is None:
        workspace = alloc_workspace(plan, dev)
    thd_indexer_topk(plan, q_i, k_i, w, idx_out, score_out, cu_seqlens_q, cu_seqlens_kv, off_q, off_k, off_out,
                     mask_type, q_causal_offset, workspace, stream)
    return idx_out, score_out


class ThdAttention(torch.autograd.Function):
    """Packed-THD attention as an autograd function: forward through
    ``thd_attn_fwd_window``, backward through ``thd_attn_bwd`` (the caller's
    metadata tensors are saved, not copied). Use :func:`thd_attention`."""

    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens_q, cu_seqlens_kv, meta: dict):
        o, stats = thd_attn_forward(q, k, v, cu_seqlens_q, cu_seqlens_kv, **meta)
        ctx.save_for_backward(q, k, v, o, stats, cu_seqlens_q, cu_seqlens_kv)
        ctx.meta = meta
        return o

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, o, stats, cu_q, cu_k = ctx.saved_tensors
        m = dict(ctx.meta)
        for name in ("o", "stats", "workspace"):   # the forward's buffers; the backward sizes its own
            m.pop(name, None)
        dq, dk, dv = thd_attn_backward(q, k, v, o, d_o.contiguous(), stats, cu_q, cu_k, **m)
        return dq, dk, dv, None, None, None


def thd_attention(q, k, v, cu_seqlens_q, cu_seqlens_kv, **meta):
    """Differentiable packed-THD attention: ``meta`` takes the keyword arguments of
    :func:`thd_attn_forward` (offsets, mask_type, q_causal_offset, window_left,
    stats_layout, softmax_scale, kernel). Returns O; gradients flow to q, k, v."""
    return ThdAttention.apply(q, k, v, cu_seqlens_q, cu_seqlens_kv, meta)
