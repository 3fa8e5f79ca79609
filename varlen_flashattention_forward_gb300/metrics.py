"""Work and traffic counts used to report throughput and roofline fractions.

pairs      number of (sequence, head, query row, key) combinations that are
           visible under the mask; the attention does 2*(d_qk + d_v) flops per
           pair (one multiply-add per element of q.k and of p.v).  With
           d_qk == d_v this is the 4 * pairs * d convention.
alg_bytes  the bytes the method must move at least once: read Q, K, V (and
           for decode the gathered rows, top-k indices and page-table rows
           those indices touch), write O and the LSE.  Re-reads of K/V by
           different query tiles are not counted.
"""
from __future__ import annotations

import numpy as np


def visible_keys_per_row(lq: int, lk: int, causal: bool, wl: int, wr: int) -> np.ndarray:
    """Count of visible keys for each query row of one sequence (closed form)."""
    i = np.arange(lq, dtype=np.int64)
    off = lk - lq
    lo = np.zeros(lq, dtype=np.int64) if wl < 0 else np.maximum(0, i + off - wl)
    hi_incl = np.full(lq, lk - 1, dtype=np.int64)
    if causal:
        hi_incl = np.minimum(hi_incl, i + off)
    if wr >= 0:
        hi_incl = np.minimum(hi_incl, i + off + wr)
    return np.maximum(0, hi_incl - lo + 1)


def varlen_pairs(lens_q, lens_k, num_heads, causal=False, window=(-1, -1)) -> int:
    wl, wr = window
    total = 0
    for lq, lk in zip(lens_q, lens_k):
        total += int(visible_keys_per_row(lq, lk, causal, wl, wr).sum())
    return total * num_heads


def varlen_flops(w) -> float:
    pairs = varlen_pairs(w.lens_q, w.lens_k, w.num_heads, w.causal, w.window)
    return 2.0 * pairs * (w.d_qk + w.d_v)


def varlen_alg_bytes(w, with_lse=None) -> float:
    with_lse = w.return_lse if with_lse is None else with_lse
    b = 2.0 * (w.total_q * w.num_heads * w.d_qk
               + w.total_k * w.num_heads_k * (w.d_qk + w.d_v)
               + w.total_q * w.num_heads * w.d_v)
    if with_lse:
        b += 4.0 * w.total_q * w.num_heads
    return b


def decode_pairs(d) -> int:
    return d.num_tokens * d.num_heads * d.topk


def decode_flops(d) -> float:
    return 2.0 * decode_pairs(d) * (576 + 512)


def decode_alg_bytes(d, with_lse=True) -> float:
    rows = d.num_tokens * d.topk * 576 * 2          # gathered cache rows
    idx = d.num_tokens * d.topk * 4                 # top-k indices
    pages = d.num_tokens * d.pages_per_token * 4    # page-table rows
    q = d.num_tokens * d.num_heads * 576 * 2
    out = d.num_tokens * d.num_heads * 512 * 2
    lse = d.num_tokens * d.num_heads * 4 if with_lse else 0
    return float(rows + idx + pages + q + out + lse)
