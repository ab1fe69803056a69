"""CPU oracle for paged split-KV GQA decode attention (fp64).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of ``bench.py`` are the only callers.  Nothing
here imports the CUDA library or anything under ``paged_split_kv_gqa_gb300``
except the seeded input generators, and the CUDA path never imports this.

Two independent implementations of the same plain definition:

* O1 -- ``ga_oracle.c`` (C, fp64, OpenMP over (row, kv head)), loaded with
  ctypes: gathers the keys of a row through its page table and evaluates
  softmax attention key by key.  This is the oracle the GPU is compared with
  and the one the CPU baseline times.
* O2 -- :func:`brute_decode` (numpy, fp64): rebuilds every row's whole
  logical sequence with vectorised fancy indexing, scores *all* positions and
  applies an explicit boolean mask built from a position comparison.  Tiny
  inputs only; it exists to pin O1.

The definition (cited from the pages by title and section):

* block-GQA: query head h reads kv head floor(h / (Hq / Hkv))
  ("visible-cx/Gemma-4-31B-CoreAI", hybrid-pf64 bundles, numerics gate).
* sliding window W for the local family, query at position L-1 sees keys
  j with (L-1) - j < W ("[Model] Gemma 4 M3 31B", Acceptance Criteria:
  boundaries 1023 / 1024 / 1025); global family sees all L keys.
* paged KV: key j of row b sits in page page_table[b][j // P], slot j % P
  ("[Model] Gemma 4 M1 12B", Description).
* softmax attention with an explicit scale, the split-KV partials merged by
  log-sum-exp ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is mandatory
  here": flash-decode split factor 8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

KV_BF16 = 0
KV_E4M3 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ga_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ga_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            c_i32, c_i64, c_p, c_d = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = c_d
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = c_d
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_key_range.argtypes = [c_i32, c_i32, c_p, c_p]
            L.oracle_key_range.restype = None
            L.oracle_logical_pages.argtypes = [c_i32, c_i32, c_i32, c_p, c_p]
            L.oracle_logical_pages.restype = None
            L.oracle_decode.argtypes = [c_p, c_p, c_p, ctypes.c_int, c_p, c_p, c_p, c_i64, c_p,
                                        c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i64, c_d,
                                        c_p, c_i32, c_i32, c_p, c_p, c_i32]
            L.oracle_decode.restype = ctypes.c_int
            L.oracle_decode_mq.argtypes = [c_p, c_p, c_p, ctypes.c_int, c_p, c_p, c_p, c_i64,
                                           c_p, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                           c_i64, c_i32, c_d, c_p, c_p, c_i32]
            L.oracle_decode_mq.restype = ctypes.c_int
            L.oracle_combine.argtypes = [c_p, c_p, c_i32, c_i32, c_p]
            L.oracle_combine.restype = c_d
            L.oracle_kv_append.argtypes = [c_p, c_p, c_p, c_p, ctypes.c_int, c_p, c_p, c_p, c_i64,
                                           c_p, c_i32, c_i32, c_i32, c_i32, c_i64]
            L.oracle_kv_append.restype = ctypes.c_int
            L.oracle_max_threads.argtypes = []
            L.oracle_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _np(a, dtype=None):
    """numpy view of a CPU tensor / array, C-contiguous (bf16 as uint16 bits)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.uint16) if hasattr(torch, "uint16") else a.view(torch.int16)
                return np.ascontiguousarray(a.numpy().view(np.uint16))
            if a.dtype == torch.float8_e4m3fn:
                return np.ascontiguousarray(a.view(torch.uint8).numpy())
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None:
        a = np.ascontiguousarray(a.astype(dtype, copy=False))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (numpy, no C)."""
    w = bits.astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return w.view(np.float32).astype(np.float64)


def key_range(L: int, W: int):
    lo, hi = ctypes.c_int32(), ctypes.c_int32()
    lib().oracle_key_range(int(L), int(W), ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def logical_pages(L: int, W: int, P: int):
    """(first logical page, page count) holding the keys a row attends."""
    f, n = ctypes.c_int32(), ctypes.c_int32()
    lib().oracle_logical_pages(int(L), int(W), int(P), ctypes.byref(f), ctypes.byref(n))
    return f.value, n.value


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


# ------------------------------------------------------------------ O1

def decode(q, k_pool, v_pool, page_table, seq_lens, *, num_kv_heads, window, scale,
           kv_dtype=KV_BF16, k_scale=None, v_scale=None, rows=None, chunk_pages=0,
           nthreads=0, return_lse=False):
    """O1: fp64 paged decode.  Returns out [nrows, Hq, D] float64 (and lse).

    q [B, Hq, D] bf16; pools [num_pages, Hkv, P, D] bf16 or e4m3 codes;
    page_table [B, stride] int32; seq_lens [B] int32; window 0 = global.
    rows: optional subset of row indices (output rows follow that order).
    chunk_pages > 0 evaluates page-aligned chunks merged by log-sum-exp.
    """
    qn = _np(q)
    assert qn.dtype == np.uint16 and qn.ndim == 3
    B, Hq, D = qn.shape
    kp, vp = _np(k_pool), _np(v_pool)
    num_pages, Hkv, P, D2 = kp.shape
    assert D2 == D and Hkv == num_kv_heads and vp.shape == kp.shape
    if kv_dtype == KV_BF16:
        assert kp.dtype == np.uint16
    else:
        assert kp.dtype == np.uint8
    pt = _np(page_table, np.int32)
    sl = _np(seq_lens, np.int32)
    ks = _np(k_scale, np.float32) if k_scale is not None else None
    vs = _np(v_scale, np.float32) if v_scale is not None else None
    if kv_dtype == KV_E4M3:
        assert ks is not None and vs is not None
    rws = _np(rows, np.int32) if rows is not None else None
    nr = len(rws) if rws is not None else B
    out = np.zeros((nr, Hq, D), dtype=np.float64)
    lse = np.zeros((nr, Hq), dtype=np.float64)
    rc = lib().oracle_decode(_ptr(qn), _ptr(kp), _ptr(vp), kv_dtype, _ptr(ks), _ptr(vs),
                             _ptr(pt), pt.shape[1], _ptr(sl), B, Hq, Hkv, D, int(window), P,
                             num_pages, float(scale), _ptr(rws), nr, int(chunk_pages),
                             _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_decode: invalid input (code {rc})")
    return (out, lse) if return_lse else out


def decode_mq(q, k_pool, v_pool, page_table, seq_lens, *, num_kv_heads, window, scale,
              kv_dtype=KV_BF16, k_scale=None, v_scale=None, nthreads=0, return_lse=False):
    """O1 multi-query decode: q [B, Hq, S, D] bf16 -> out [B, Hq, S, D] float64.

    Query i of row b sits at position L_b - S + i and attends the keys of a
    one-query row of length L_b - S + i + 1 (causal inside the chunk; the
    sliding window ends at its own position).
    """
    qn = _np(q)
    assert qn.dtype == np.uint16 and qn.ndim == 4
    B, Hq, S, D = qn.shape
    kp, vp = _np(k_pool), _np(v_pool)
    num_pages, Hkv, P, D2 = kp.shape
    assert D2 == D and Hkv == num_kv_heads and vp.shape == kp.shape
    assert kp.dtype == (np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    pt = _np(page_table, np.int32)
    sl = _np(seq_lens, np.int32)
    ks = _np(k_scale, np.float32) if k_scale is not None else None
    vs = _np(v_scale, np.float32) if v_scale is not None else None
    if kv_dtype == KV_E4M3:
        assert ks is not None and vs is not None
    out = np.zeros((B, Hq, S, D), dtype=np.float64)
    lse = np.zeros((B, Hq, S), dtype=np.float64)
    rc = lib().oracle_decode_mq(_ptr(qn), _ptr(kp), _ptr(vp), kv_dtype, _ptr(ks), _ptr(vs),
                                _ptr(pt), pt.shape[1], _ptr(sl), B, Hq, Hkv, D, int(window), P,
                                num_pages, S, float(scale), _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_decode_mq: invalid input (code {rc})")
    return (out, lse) if return_lse else out


def combine(partial_o, partial_lse):
    """LSE merge of S partials: partial_o [S, D], partial_lse [S] -> (o [D], lse)."""
    po = np.ascontiguousarray(partial_o, dtype=np.float64)
    pl = np.ascontiguousarray(partial_lse, dtype=np.float64)
    S, D = po.shape
    o = np.zeros(D, dtype=np.float64)
    lse = lib().oracle_combine(_ptr(po), _ptr(pl), S, D, _ptr(o))
    return o, lse


def kv_append(k_new, v_new, k_pool, v_pool, page_table, positions, *, kv_dtype=KV_BF16,
              k_scale=None, v_scale=None):
    """O1 append on numpy copies.  Returns the updated (k_pool, v_pool) arrays."""
    kn, vn = _np(k_new), _np(v_new)
    kp, vp = _np(k_pool).copy(), _np(v_pool).copy()
    num_pages, Hkv, P, D = kp.shape
    B = kn.shape[0]
    pt = _np(page_table, np.int32)
    pos = _np(positions, np.int32)
    ks = _np(k_scale, np.float32) if k_scale is not None else None
    vs = _np(v_scale, np.float32) if v_scale is not None else None
    rc = lib().oracle_kv_append(_ptr(kn), _ptr(vn), _ptr(kp), _ptr(vp), kv_dtype, _ptr(ks),
                                _ptr(vs), _ptr(pt), pt.shape[1], _ptr(pos), B, Hkv, D, P,
                                num_pages)
    if rc != 0:
        raise ValueError(f"oracle_kv_append: invalid input (code {rc})")
    return kp, vp


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ------------------------------------------------------------------ O2

def brute_decode(q, k_pool, v_pool, page_table, seq_lens, *, num_kv_heads, window, scale,
                 kv_dtype=KV_BF16, k_scale=None, v_scale=None):
    """O2: dense masked softmax in numpy fp64 (tiny inputs only).

    For each row the whole logical sequence 0..L-1 is materialised through the
    page table with one fancy-indexing gather; scores are taken for every
    position and a boolean mask (pos < L) & (L-1 - pos < W) selects the keys.
    Dequantisation of e4m3 codes uses a 256-entry table built from the bit
    fields, independent of the C decoder.
    """
    qn = bf16_bits_to_f64(_np(q))
    kp, vp = _np(k_pool), _np(v_pool)
    num_pages, Hkv, P, D = kp.shape
    if kv_dtype == KV_BF16:
        Kf, Vf = bf16_bits_to_f64(kp), bf16_bits_to_f64(vp)
    else:
        table = _e4m3_table_numpy()
        ks = _np(k_scale, np.float32).astype(np.float64)
        vs = _np(v_scale, np.float32).astype(np.float64)
        Kf = table[kp] * ks[None, :, None, None]
        Vf = table[vp] * vs[None, :, None, None]
    pt = _np(page_table, np.int64)
    sl = _np(seq_lens, np.int64)
    B, Hq, _ = qn.shape
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(sl[b])
        if L <= 0:
            continue
        pos = np.arange(L)
        phys = pt[b, pos // P]
        slot = pos % P
        mask = (pos <= L - 1)
        if window > 0:
            mask &= (L - 1 - pos) < window
        for h in range(Hq):
            c = h // g
            K = Kf[phys, c, slot, :]          # [L, D]
            V = Vf[phys, c, slot, :]
            s = scale * (K @ qn[b, h])
            s = np.where(mask, s, -np.inf)
            w = np.exp(s - s.max())
            out[b, h] = (w[:, None] * V).sum(0) / w.sum()
    return out


def brute_decode_mq(q, k_pool, v_pool, page_table, seq_lens, *, num_kv_heads, window, scale):
    """O2 multi-query (bf16 pools, tiny inputs): q [B, Hq, S, D] -> [B, Hq, S, D].

    The whole row 0..L-1 is materialised; query i at position t = L - S + i
    keeps key j iff j <= t (causal) and t - j < window (sliding family).
    """
    qn = bf16_bits_to_f64(_np(q))
    kp, vp = _np(k_pool), _np(v_pool)
    num_pages, Hkv, P, D = kp.shape
    Kf, Vf = bf16_bits_to_f64(kp), bf16_bits_to_f64(vp)
    pt = _np(page_table, np.int64)
    sl = _np(seq_lens, np.int64)
    B, Hq, S, _ = qn.shape
    g = Hq // Hkv
    out = np.zeros((B, Hq, S, D), dtype=np.float64)
    for b in range(B):
        L = int(sl[b])
        if L <= 0:
            continue
        pos = np.arange(L)
        phys = pt[b, pos // P]
        slot = pos % P
        for h in range(Hq):
            c = h // g
            K = Kf[phys, c, slot, :]
            V = Vf[phys, c, slot, :]
            for i in range(S):
                t = L - S + i
                mask = pos <= t
                if window > 0:
                    mask &= (t - pos) < window
                if not mask.any():
                    continue
                s = np.where(mask, scale * (K @ qn[b, h, i]), -np.inf)
                w = np.exp(s - s.max())
                out[b, h, i] = (w[:, None] * V).sum(0) / w.sum()
    return out


def _e4m3_table_numpy() -> np.ndarray:
    codes = np.arange(256)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = (codes & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = sign * val
    val[(e == 15) & ((codes & 7) == 7)] = np.nan
    return val
