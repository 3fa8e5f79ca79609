"""Plain fp64 CPU oracle for the attention forward pass.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product package never imports it.
It shares no code with the CUDA path.  The arithmetic lives in
``attention_oracle.c`` (plain C, fp64, OpenMP over rows); this module only
compiles it with gcc and marshals arrays through ctypes.

Functions:
  varlen_attention(...)   -> (out [rows, d_v] f64, lse [rows] f64)
  sparse_mla_decode(...)  -> (out [rows, 512] f64, lse [rows] f64)
  merge_states(...)       -> (out [rows, d] f64, lse [rows] f64)
Rows are (token, head) pairs flattened as token * H + head.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(library routines, closed forms, invariants, hand-enumerated golden masks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attention_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_varlen_attention.argtypes = [
                p, p, p, p, p, i32, i32, i32, i32, i32, f64, i32, i32, i32,
                i64, p, p, p, i32]
            lib.oracle_varlen_attention.restype = i32
            lib.oracle_sparse_mla_decode.argtypes = [
                p, p, p, p, i32, i32, i32, i32, i32, i32, f64, i64, p, p, p,
                i32]
            lib.oracle_sparse_mla_decode.restype = i32
            lib.oracle_merge_states.argtypes = [p, p, p, p, i64, i32, p, p]
            lib.oracle_merge_states.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def _bf16_bits(x) -> np.ndarray:
    """bf16 torch tensor (or uint16 array of bf16 bits) -> contiguous uint16."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(
        x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale,
                     causal=False, window_left=-1, window_right=-1,
                     rows=None, threads=0):
    """fp64 attention over packed sequences.

    q [total_q, H, d_qk], k [total_k, H_k, d_qk], v [total_k, H_k, d_v] (bf16).
    rows: optional int64 array of flattened token*H + head ids.
    Returns (out [rows, d_v], lse [rows]) as float64 numpy arrays.
    """
    lib = _load()
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    assert qb.ndim == 3 and kb.ndim == 3 and vb.ndim == 3
    total_q, H, d_qk = qb.shape
    _, H_k, d_v = vb.shape
    assert kb.shape[1] == H_k and kb.shape[2] == d_qk
    batch = cq.shape[0] - 1
    if rows is None:
        n = total_q * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    out = np.zeros((n, d_v), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_varlen_attention(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(cq), _ptr(ck), batch, H, H_k, d_qk,
        d_v, float(softmax_scale), int(bool(causal)), int(window_left),
        int(window_right), n, None if rows_arr is None else _ptr(rows_arr),
        _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_varlen_attention failed with status {rc}")
    return out, lse


def sparse_mla_decode(q, kv_cache, page_table, topk_idx, softmax_scale,
                      page_size=64, rows=None, threads=0):
    """fp64 sparse-MLA decode.

    q [T, H, 576] bf16, kv_cache [num_pages, page_size, 576] bf16,
    page_table [T, max_pages] int32, topk_idx [T, topk] int32.
    Returns (out [rows, 512], lse [rows]) as float64 numpy arrays.
    """
    lib = _load()
    qb, cb = _bf16_bits(q), _bf16_bits(kv_cache)
    pt, ti = _i32(page_table), _i32(topk_idx)
    T, H, dq = qb.shape
    assert dq == 576 and cb.shape[-1] == 576 and cb.shape[1] == page_size
    num_pages = cb.shape[0]
    max_pages = pt.shape[1]
    topk = ti.shape[1]
    if rows is None:
        n = T * H
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    out = np.zeros((n, 512), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_sparse_mla_decode(
        _ptr(qb), _ptr(cb), _ptr(pt), _ptr(ti), T, H, topk, num_pages,
        max_pages, page_size, float(softmax_scale), n,
        None if rows_arr is None else _ptr(rows_arr), _ptr(out), _ptr(lse),
        int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_sparse_mla_decode failed with status {rc}")
    return out, lse


def merge_states(o_a, lse_a, o_b, lse_b):
    """LSE-weighted merge of two partial results over disjoint key sets.

    o_*: [rows, d] float64 arrays (or bf16 torch tensors, widened exactly),
    lse_*: [rows].  Returns (out [rows, d], lse [rows]) float64.
    """
    lib = _load()

    def f64(x):
        if not isinstance(x, np.ndarray):
            x = x.detach().cpu().double().numpy()
        return np.ascontiguousarray(x, dtype=np.float64)
    oa, ob, la, lb = f64(o_a), f64(o_b), f64(lse_a).reshape(-1), f64(lse_b).reshape(-1)
    rows = la.shape[0]
    oa, ob = oa.reshape(rows, -1), ob.reshape(rows, -1)
    d = oa.shape[1]
    out = np.zeros((rows, d), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    rc = lib.oracle_merge_states(_ptr(oa), _ptr(la), _ptr(ob), _ptr(lb), rows, d,
                                 _ptr(out), _ptr(lse))
    if rc != 0:
        raise RuntimeError(f"oracle_merge_states failed with status {rc}")
    return out, lse
