"""GB300 (sm_103a) variable-length attention forward -- Python binding.

Thin ctypes marshalling over the C ABI of ``libfa_gb300.so`` (declared in
``include/fa_gb300.h``).  Every step of the computation runs in the library's
CUDA kernels; this module only checks tensor shapes/dtypes, passes raw device
pointers and sizes, and turns status codes into exceptions.  There is no CPU
or PyTorch fallback: if the library is missing, the entry points raise.

Entry points (same names as the C ABI):
  fa_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                max_seqlen_k, softmax_scale, causal=False, window_left=-1,
                window_right=-1, out=None, lse=None, return_lse=False,
                stream=None)
  fa_varlen_fwd_plan(batch, total_q, total_k, num_heads, num_heads_k, d_qk, d_v,
                     max_seqlen_q=0, max_seqlen_k=0, causal=False, window_left=-1,
                     window_right=-1)
  fa_sparse_mla_decode(q, kv_cache, page_table, topk_idx, softmax_scale,
                       out=None, lse=None, return_lse=False, stream=None)
  fa_sparse_mla_decode_plan(num_tokens, num_heads, topk)
  fa_sparse_mla_decode_noalloc(q, kv_cache, page_table, topk_idx, softmax_scale,
                               out, lse=None, stream=None)
  fa_merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse,
                       out=None, out_lse=None, stream=None)
  fa_get_device_status()
  fa_set_wait_limit_ns(ns)
"""
from __future__ import annotations

import ctypes
import os

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ARCH = 3
FA_ERR_LAUNCH = 4
FA_ERR_DEVICE_TIMEOUT = 5
FA_ERR_SCRATCH = 6
NOALLOC_SCRATCH_BYTES = 48 << 20  # FA_NOALLOC_SCRATCH_BYTES

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

# Exported C symbols (kept in sync with include/fa_gb300.h; a CPU test checks).
EXPORTS = ("fa_varlen_fwd", "fa_varlen_fwd_plan", "fa_varlen_fwd_strided", "fa_sparse_mla_decode",
           "fa_sparse_mla_decode_plan", "fa_sparse_mla_decode_noalloc", "fa_merge_attn_states",
           "fa_get_device_status", "fa_set_wait_limit_ns", "fa_status_string")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load_library():
    """Loads libfa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_varlen_fwd.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32,
                                  i32, i32, i32, f32, i32, i32, i32, p, p, p]
    lib.fa_varlen_fwd.restype = i32
    i64 = ctypes.c_longlong
    lib.fa_varlen_fwd_strided.argtypes = [p, i64, i64, p, i64, i64, p, i64, i64, p, p, i32,
                                          i32, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                          i32, i32, p, p, p]
    lib.fa_varlen_fwd_strided.restype = i32
    lib.fa_sparse_mla_decode.argtypes = [p, p, p, p, i32, i32, i32, i32, i32,
                                         f32, p, p, p]
    lib.fa_sparse_mla_decode.restype = i32
    pi = ctypes.POINTER(i32)
    lib.fa_varlen_fwd_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                       i32, pi, pi, pi]
    lib.fa_varlen_fwd_plan.restype = i32
    lib.fa_sparse_mla_decode_plan.argtypes = [i32, i32, i32, ctypes.POINTER(i32),
                                              ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_sparse_mla_decode_plan.restype = i32
    lib.fa_sparse_mla_decode_noalloc.argtypes = [p, p, p, p, i32, i32, i32, i32, i32,
                                                 f32, p, p, p]
    lib.fa_sparse_mla_decode_noalloc.restype = i32
    lib.fa_merge_attn_states.argtypes = [p, p, p, p, p, p, i32, i32, i32, p]
    lib.fa_merge_attn_states.restype = i32
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_wait_limit_ns.restype = i32
    lib.fa_get_device_status.argtypes = []
    lib.fa_get_device_status.restype = i32
    lib.fa_status_string.argtypes = [i32]
    lib.fa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().fa_status_string(int(status)).decode()
    except Exception:  # library unavailable: still give a readable message
        return f"status {status}"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, ndim, view=False):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if view:
        # A strided view is passed as (pointer, row stride, head stride); the
        # library checks the strides, the innermost dimension must be dense.
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous last dimension")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q=0,
                  max_seqlen_k=0, softmax_scale=None, causal=False,
                  window_left=-1, window_right=-1, out=None, lse=None,
                  return_lse=False, stream=None):
    """Varlen attention forward; see fa_varlen_fwd in include/fa_gb300.h.

    q [total_q, H, d_qk], k [total_k, H_k, d_qk], v [total_k, H_k, d_v] bf16
    CUDA tensors; cu_seqlens_* int32 [batch+1] CUDA tensors.  Returns out
    [total_q, H, d_v] bf16, or (out, lse [H, total_q] fp32) if an lse buffer
    is given or return_lse is set.  q, k and v may be strided views with a
    contiguous last dimension (for example V taken out of a combined
    [tokens, heads, nope + v] buffer); they then go through
    fa_varlen_fwd_strided.
    """
    import torch
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, torch.bfloat16, 3, view=True)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    total_q, H, d_qk = q.shape
    total_k, H_k, d_v = v.shape
    if k.shape[0] != total_k or k.shape[1] != H_k or k.shape[2] != d_qk:
        raise ValueError(f"k shape {tuple(k.shape)} inconsistent with q/v")
    batch = cu_seqlens_q.shape[0] - 1
    if cu_seqlens_k.shape[0] != batch + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
    if softmax_scale is None:
        softmax_scale = d_qk ** -0.5
    if out is None:
        out = torch.empty((total_q, H, d_v), dtype=torch.bfloat16, device=q.device)
    else:
        _check(out, "out", torch.bfloat16, 3)
    if lse is None and return_lse:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2)
    if q.is_contiguous() and k.is_contiguous() and v.is_contiguous():
        st = lib.fa_varlen_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            batch, total_q, total_k, H, H_k, d_qk, d_v, int(max_seqlen_q),
            int(max_seqlen_k), float(softmax_scale), int(bool(causal)),
            int(window_left), int(window_right), _ptr(out), _ptr(lse),
            _stream_ptr(stream))
    else:
        st = lib.fa_varlen_fwd_strided(
            _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1),
            _ptr(v), v.stride(0), v.stride(1), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            batch, total_q, total_k, H, H_k, d_qk, d_v, int(max_seqlen_q),
            int(max_seqlen_k), float(softmax_scale), int(bool(causal)),
            int(window_left), int(window_right), _ptr(out), _ptr(lse),
            _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_varlen_fwd")
    return (out, lse) if lse is not None else out


def fa_sparse_mla_decode(q, kv_cache, page_table, topk_idx, softmax_scale=None,
                         out=None, lse=None, return_lse=False, stream=None):
    """Sparse-MLA decode; see fa_sparse_mla_decode in include/fa_gb300.h.

    q [T, H, 576] bf16, kv_cache [num_pages, 64, 576] bf16, page_table
    [T, max_pages] int32, topk_idx [T, topk] int32 (CUDA tensors).  Returns
    out [T, H, 512] bf16, or (out, lse [H, T] fp32).
    """
    import torch
    lib = load_library()
    _check(q, "q", torch.bfloat16, 3)
    _check(kv_cache, "kv_cache", torch.bfloat16, 3)
    _check(page_table, "page_table", torch.int32, 2)
    _check(topk_idx, "topk_idx", torch.int32, 2)
    T, H, dq = q.shape
    if dq != 576 or kv_cache.shape[1] != 64 or kv_cache.shape[2] != 576:
        raise ValueError("q must be [T, H, 576] and kv_cache [pages, 64, 576]")
    if page_table.shape[0] != T or topk_idx.shape[0] != T:
        raise ValueError("page_table / topk_idx must have one row per token")
    if softmax_scale is None:
        softmax_scale = 576 ** -0.5
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    else:
        _check(out, "out", torch.bfloat16, 3)
    if lse is None and return_lse:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2)
    st = lib.fa_sparse_mla_decode(
        _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(topk_idx), T, H,
        topk_idx.shape[1], kv_cache.shape[0], page_table.shape[1],
        float(softmax_scale), _ptr(out), _ptr(lse), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_sparse_mla_decode")
    return (out, lse) if lse is not None else out


def fa_varlen_fwd_plan(batch, total_q, total_k, num_heads, num_heads_k, d_qk, d_v,
                       max_seqlen_q=0, max_seqlen_k=0, causal=False, window_left=-1,
                       window_right=-1):
    """(grid, split, heads_per_tile) of an fa_varlen_fwd call of these sizes
    on the current device: split > 1 means split-KV in clusters of `split`
    CTAs, heads_per_tile > 1 GQA head-group packing; see fa_varlen_fwd_plan
    in include/fa_gb300.h."""
    lib = load_library()
    g, s, p = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = lib.fa_varlen_fwd_plan(int(batch), int(total_q), int(total_k), int(num_heads),
                                int(num_heads_k), int(d_qk), int(d_v), int(max_seqlen_q),
                                int(max_seqlen_k), int(bool(causal)), int(window_left),
                                int(window_right), ctypes.byref(g), ctypes.byref(s),
                                ctypes.byref(p))
    if st != FA_OK:
        raise FaError(st, "fa_varlen_fwd_plan")
    return g.value, s.value, p.value


def fa_sparse_mla_decode_plan(num_tokens, num_heads, topk):
    """(launches, workspace_bytes) of a decode call of this size on the
    current device; see fa_sparse_mla_decode_plan in include/fa_gb300.h."""
    lib = load_library()
    n = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    st = lib.fa_sparse_mla_decode_plan(int(num_tokens), int(num_heads), int(topk),
                                       ctypes.byref(n), ctypes.byref(b))
    if st != FA_OK:
        raise FaError(st, "fa_sparse_mla_decode_plan")
    return n.value, b.value


def fa_sparse_mla_decode_noalloc(q, kv_cache, page_table, topk_idx, softmax_scale, out,
                                 lse=None, stream=None):
    """fa_sparse_mla_decode_noalloc (include/fa_gb300.h): the same decode with
    no device allocation, by the library or here.  `out` [T, H, 512] bf16 and
    (optionally) `lse` [H, T] fp32 are caller-provided.  Overlapping calls on
    one device race on the library's fixed scratch; the caller orders them."""
    import torch
    lib = load_library()
    _check(q, "q", torch.bfloat16, 3)
    _check(kv_cache, "kv_cache", torch.bfloat16, 3)
    _check(page_table, "page_table", torch.int32, 2)
    _check(topk_idx, "topk_idx", torch.int32, 2)
    _check(out, "out", torch.bfloat16, 3)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2)
    T, H, dq = q.shape
    if dq != 576 or kv_cache.shape[1] != 64 or kv_cache.shape[2] != 576:
        raise ValueError("q must be [T, H, 576] and kv_cache [pages, 64, 576]")
    if page_table.shape[0] != T or topk_idx.shape[0] != T or tuple(out.shape) != (T, H, 512):
        raise ValueError("page_table / topk_idx / out must have one row per token")
    st = lib.fa_sparse_mla_decode_noalloc(
        _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(topk_idx), T, H,
        topk_idx.shape[1], kv_cache.shape[0], page_table.shape[1],
        float(softmax_scale), _ptr(out), _ptr(lse), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_sparse_mla_decode_noalloc")
    return out


def fa_merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse, out=None,
                         out_lse=None, stream=None):
    """LSE-weighted merge; see fa_merge_attn_states in include/fa_gb300.h.

    *_out bf16 [T, H, d], *_lse fp32 [H, T] CUDA tensors.  Returns (out, out_lse).
    """
    import torch
    lib = load_library()
    for name, t in (("prefix_out", prefix_out), ("suffix_out", suffix_out)):
        _check(t, name, torch.bfloat16, 3)
    for name, t in (("prefix_lse", prefix_lse), ("suffix_lse", suffix_lse)):
        _check(t, name, torch.float32, 2)
    T, H, d = prefix_out.shape
    if tuple(suffix_out.shape) != (T, H, d) or tuple(prefix_lse.shape) != (H, T) \
            or tuple(suffix_lse.shape) != (H, T):
        raise ValueError("merge inputs must be [T, H, d] outputs and [H, T] LSEs")
    if out is None:
        out = torch.empty_like(prefix_out)
    if out_lse is None:
        out_lse = torch.empty_like(prefix_lse)
    st = lib.fa_merge_attn_states(_ptr(out), _ptr(out_lse), _ptr(prefix_out), _ptr(prefix_lse),
                                  _ptr(suffix_out), _ptr(suffix_lse), T, H, d,
                                  _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_merge_attn_states")
    return out, out_lse


def fa_set_wait_limit_ns(ns: int) -> None:
    """Time limit of the kernels' pipeline waits for later launches (0 = the
    default of 4 s); a test hook, see fa_set_wait_limit_ns in
    include/fa_gb300.h."""
    load_library().fa_set_wait_limit_ns(int(ns))


def fa_get_device_status() -> int:
    """Reads and clears the device status word (synchronises the device)."""
    return int(load_library().fa_get_device_status())
