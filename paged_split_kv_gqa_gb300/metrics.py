"""Algorithmic byte and token counts of one decode-attention launch.

These are what the method must move through HBM, independent of how a kernel
moves it: every attended key and value once, q in, the output out, the page
table entries read, seq_lens, and the fp8 scales.  Workspace traffic of a
split launch is not algorithmic and is reported separately.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """K and V bytes one layer stores for one token (all kv heads)."""
    return 2 * num_kv_heads * head_dim * bytes_per_elem


def attended_keys(seq_lens, window: int) -> np.ndarray:
    """Keys each row's query attends: min(L, W) for a window, else L."""
    L = np.maximum(np.asarray(seq_lens, dtype=np.int64), 0)
    return np.minimum(L, window) if window > 0 else L


def pages_read(seq_lens, window: int, page_size: int) -> np.ndarray:
    L = np.maximum(np.asarray(seq_lens, dtype=np.int64), 0)
    lo = np.maximum(L - window, 0) if window > 0 else np.zeros_like(L)
    return np.where(L > 0, (L - 1) // page_size - lo // page_size + 1, 0)


def union_window(window: int, q_len: int) -> int:
    """Window of the keys any of a row's q_len queries (its last q_len
    positions, each with its own window) attends; 0 (global) stays 0."""
    return window + q_len - 1 if window > 0 else 0


def decode_bytes(seq_lens, *, num_q_heads, num_kv_heads, head_dim, window, page_size,
                 kv_bytes_per_elem, kv_alias=False, q_len=1) -> int:
    """Algorithmic HBM bytes of one decode launch over a batch (K == V one
    pool: each attended key row is read once).  With q_len queries per row
    the keys are those of the union of their windows, read once, and q / out
    carry q_len rows per head."""
    B = len(seq_lens)
    window = union_window(window, q_len)
    n = int(attended_keys(seq_lens, window).sum())
    kv = n * kv_bytes_per_token(num_kv_heads, head_dim, kv_bytes_per_elem)
    if kv_alias:
        kv //= 2
    qo = 2 * B * num_q_heads * q_len * head_dim * 2
    table = 4 * int(pages_read(seq_lens, window, page_size).sum())
    scales = 8 * num_kv_heads if kv_bytes_per_elem == 1 else 0
    return int(kv + qo + table + 4 * B + scales)


def append_bytes(batch, *, num_kv_heads, head_dim, kv_bytes_per_elem) -> int:
    """Algorithmic bytes of one append: new K,V in (bf16), pool slots out,
    one page-table entry and one position per row."""
    return int(batch * num_kv_heads * head_dim * (2 * 2 + 2 * kv_bytes_per_elem) + 8 * batch)
