"""Thin ctypes binding of libga.so (the C ABI declared in include/ga.h).

Argument marshalling only: tensors become device pointers and sizes, the
current torch CUDA stream becomes the launch stream, and a nonzero status
becomes :class:`GAError`.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  Importing this module fails if
libga.so has not been built (``__graft_entry__.build()`` or
``python -m paged_split_kv_gqa_gb300._build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import _build

GA_OK = 0
GA_ERR_INVALID_ARG = 1
GA_ERR_UNSUPPORTED = 2
GA_ERR_WORKSPACE_TOO_SMALL = 3
GA_ERR_CUDA = 4
GA_ERR_DEVICE_CHECK = 5

GA_KV_BF16 = 0
GA_KV_E4M3 = 1

GA_DEVERR_PAGE_ID = 1
GA_DEVERR_SEQ_LEN = 2
GA_DEVERR_CAPACITY = 4
GA_DEVERR_Q_RANGE = 8
GA_DEVERR_TIMEOUT = 16
GA_DEVERR_POSITION = 32

GA_SPLIT_NONE = 0
GA_SPLIT_COUNT = 1
GA_SPLIT_CHUNK = 2
GA_SCHEDULE_ROUND_ROBIN = 0
GA_SCHEDULE_ROWS_BY_SIZE = 1
GA_PLAN_TOUCH_LOG = 1
GA_PLAN_EXTERNAL_COMBINE = 2
GA_PLAN_TEST_WAIT_TIMEOUT = 4
GA_PLAN_TENSOR_CORE_UNITS = 8
GA_PLAN_COLUMN_PARALLEL_UNITS = 16
GA_PLAN_KV_E4M3 = 32
PAGE_SIZE = 16
MAX_Q_LEN = 64


class GAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)}")


class ga_plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "mode", "splits", "chunk_pages", "batch", "num_q_heads", "num_kv_heads", "head_dim",
        "window", "page_size", "grid", "flags", "touch_stride", "q_len", "col_tile")] + [
        (n, ctypes.c_int64) for n in ("row_chunks", "units", "workspace_bytes",
                                       "partial_o_offset", "partial_lse_offset",
                                       "touch_log_offset")] + [
        (n, ctypes.c_int32) for n in ("kv_heads_per_unit", "schedule")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libga.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    i32, i64, p, f32, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER(ga_plan)
    lib.ga_plan_splits.argtypes = [p, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, P]
    lib.ga_plan_splits_mq.argtypes = [p, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, P]
    lib.ga_kv_append.argtypes = [p, p, p, p, i32, p, p, p, i64, p, i32, i32, i32, i32, i64, p, p]
    lib.ga_decode_local_hd256.argtypes = [p, p, p, i32, p, p, p, i64, p, i32, i32, i32, i32, i32,
                                          i64, f32, P, p, sz, p, p, p]
    lib.ga_decode_global_hd512.argtypes = [p, p, p, i32, p, p, p, i64, p, i32, i32, i32, i32,
                                           i64, f32, P, p, sz, p, p, p]
    lib.ga_decode_local_hd256_append.argtypes = [p, p, p, p, p, i32, p, p, p, i64, p, i32, i32,
                                                 i32, i32, i32, i64, f32, P, p, sz, p, p, p]
    lib.ga_decode_global_hd512_append.argtypes = [p, p, p, p, p, i32, p, p, p, i64, p, i32, i32,
                                                  i32, i32, i64, f32, P, p, sz, p, p, p]
    lib.ga_splitkv_combine.argtypes = [p, p, P, p, i64, p, p, p]
    lib.ga_decode_global_hd512_noalloc.argtypes = [p, p, p, i32, p, p, p, i64, p, i32, i32, i32,
                                                   i32, i64, f32, P, p, p, p]
    for fn in ("ga_plan_splits", "ga_plan_splits_mq", "ga_kv_append", "ga_decode_local_hd256",
               "ga_decode_global_hd512", "ga_splitkv_combine", "ga_check_error_word",
               "ga_decode_global_hd512_noalloc", "ga_read_stream",
               "ga_decode_local_hd256_append", "ga_decode_global_hd512_append"):
        getattr(lib, fn).restype = ctypes.c_int
    lib.ga_read_stream.argtypes = [p, i64, p, p]
    lib.ga_check_error_word.argtypes = [i32]
    lib.ga_strerror.argtypes = [ctypes.c_int]
    lib.ga_strerror.restype = ctypes.c_char_p
    lib.ga_version.argtypes = []
    lib.ga_version.restype = i32
    return lib


_lib = _load()
lib = _lib


def strerror(status: int) -> str:
    return _lib.ga_strerror(int(status)).decode()


def ga_version() -> int:
    return int(_lib.ga_version())


def _check(status: int, where: str):
    if status != GA_OK:
        raise GAError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libga must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _kv_dtype(pool: torch.Tensor) -> int:
    if pool.dtype == torch.bfloat16:
        return GA_KV_BF16
    if pool.dtype in (torch.uint8, torch.float8_e4m3fn):
        return GA_KV_E4M3
    raise TypeError(f"KV pool dtype {pool.dtype} is not bf16 or E4M3 codes")


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


# ------------------------------------------------------------------ entry points

def ga_plan_splits(seq_lens_host: Sequence[int], *, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, window: int, page_size: int = PAGE_SIZE,
                   num_sms: Optional[int] = None, requested_splits: int = 0,
                   fixed_chunk_tokens: int = 0, flags: int = 0, q_len: int = 1) -> ga_plan:
    """Host-only planner (no CUDA call unless num_sms is looked up).  q_len > 1
    plans a multi-query decode (ga_plan_splits_mq)."""
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32).reshape(-1))
    if num_sms is None:
        num_sms = globals()["num_sms"]()
    plan = ga_plan()
    if q_len == 1:
        st = _lib.ga_plan_splits(lens.ctypes.data_as(ctypes.c_void_p), len(lens), num_q_heads,
                                 num_kv_heads, head_dim, window, page_size, num_sms,
                                 requested_splits, fixed_chunk_tokens, flags, ctypes.byref(plan))
        _check(st, "ga_plan_splits")
    else:
        st = _lib.ga_plan_splits_mq(lens.ctypes.data_as(ctypes.c_void_p), len(lens), num_q_heads,
                                    num_kv_heads, head_dim, window, page_size, q_len, num_sms,
                                    requested_splits, fixed_chunk_tokens, flags,
                                    ctypes.byref(plan))
        _check(st, "ga_plan_splits_mq")
    return plan


def workspace_for(plan: ga_plan, device=None) -> Optional[torch.Tensor]:
    """A caller-side workspace buffer of plan.workspace_bytes (None if 0)."""
    if plan.workspace_bytes == 0:
        return None
    return torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=device or "cuda")


def ga_kv_append(k_new, v_new, k_pool, v_pool, page_table, positions, *, k_scale=None,
                 v_scale=None, err_word=None, stream=None):
    B, Hkv, D = k_new.shape
    st = _lib.ga_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                           _kv_dtype(k_pool), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
                           page_table.shape[1], _ptr(positions), B, Hkv, D, k_pool.shape[2],
                           k_pool.shape[0], _ptr(err_word), _stream(stream))
    _check(st, "ga_kv_append")


def _decode(fn, name, q, k_pool, v_pool, page_table, seq_lens, *, window, scale, plan,
            workspace, out, k_scale, v_scale, err_word, stream):
    # q / out: [B, Hq, D], or [B, Hq, S, D] with S = plan.q_len query tokens per row
    if q.dim() == 4:
        B, Hq, S, D = q.shape
    else:
        (B, Hq, D), S = q.shape, 1
    if S != plan.q_len or out.shape != q.shape:
        raise GAError(GA_ERR_INVALID_ARG, f"{name}: q / out shape vs plan.q_len = {plan.q_len}")
    Hkv = k_pool.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(q), _ptr(k_pool), _ptr(v_pool), _kv_dtype(k_pool), _ptr(k_scale), _ptr(v_scale),
            _ptr(page_table), page_table.shape[1], _ptr(seq_lens), B, Hq, Hkv]
    if window is not None:
        args.append(window)
    args += [k_pool.shape[2], k_pool.shape[0], float(scale), ctypes.byref(plan), _ptr(workspace),
             ws_bytes, _ptr(out), _ptr(err_word), _stream(stream)]
    _check(fn(*args), name)
    return out


def ga_decode_local_hd256(q, k_pool, v_pool, page_table, seq_lens, *, window, scale, plan,
                          workspace=None, out=None, k_scale=None, v_scale=None, err_word=None,
                          stream=None):
    if out is None:
        out = torch.empty_like(q)
    return _decode(_lib.ga_decode_local_hd256, "ga_decode_local_hd256", q, k_pool, v_pool,
                   page_table, seq_lens, window=window, scale=scale, plan=plan,
                   workspace=workspace, out=out, k_scale=k_scale, v_scale=v_scale,
                   err_word=err_word, stream=stream)


def ga_decode_global_hd512(q, k_pool, v_pool, page_table, seq_lens, *, scale, plan,
                           workspace=None, out=None, k_scale=None, v_scale=None, err_word=None,
                           stream=None):
    if out is None:
        out = torch.empty_like(q)
    return _decode(_lib.ga_decode_global_hd512, "ga_decode_global_hd512", q, k_pool, v_pool,
                   page_table, seq_lens, window=None, scale=scale, plan=plan,
                   workspace=workspace, out=out, k_scale=k_scale, v_scale=v_scale,
                   err_word=err_word, stream=stream)


def _decode_append(fn, name, k_new, v_new, q, k_pool, v_pool, page_table, seq_lens, *, window,
                   scale, plan, workspace, out, k_scale, v_scale, err_word, stream):
    B, Hq, D = q.shape
    if plan.q_len != 1 or out.shape != q.shape or k_new.shape != (B, k_pool.shape[1], D) \
            or v_new.shape != k_new.shape:
        raise GAError(GA_ERR_INVALID_ARG, f"{name}: q / out / k_new / v_new shapes")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(k_new), _ptr(v_new), _ptr(q), _ptr(k_pool), _ptr(v_pool), _kv_dtype(k_pool),
            _ptr(k_scale), _ptr(v_scale), _ptr(page_table), page_table.shape[1], _ptr(seq_lens),
            B, Hq, k_pool.shape[1]]
    if window is not None:
        args.append(window)
    args += [k_pool.shape[2], k_pool.shape[0], float(scale), ctypes.byref(plan), _ptr(workspace),
             ws_bytes, _ptr(out), _ptr(err_word), _stream(stream)]
    _check(fn(*args), name)
    return out


def ga_decode_local_hd256_append(k_new, v_new, q, k_pool, v_pool, page_table, seq_lens, *,
                                 window, scale, plan, workspace=None, out=None, k_scale=None,
                                 v_scale=None, err_word=None, stream=None):
    """Append this step's token (at seq_lens - 1) and decode, in one launch."""
    if out is None:
        out = torch.empty_like(q)
    return _decode_append(_lib.ga_decode_local_hd256_append, "ga_decode_local_hd256_append",
                          k_new, v_new, q, k_pool, v_pool, page_table, seq_lens, window=window,
                          scale=scale, plan=plan, workspace=workspace, out=out, k_scale=k_scale,
                          v_scale=v_scale, err_word=err_word, stream=stream)


def ga_decode_global_hd512_append(k_new, v_new, q, k_pool, v_pool, page_table, seq_lens, *,
                                  scale, plan, workspace=None, out=None, k_scale=None,
                                  v_scale=None, err_word=None, stream=None):
    """Append this step's token (at seq_lens - 1) and decode, in one launch."""
    if out is None:
        out = torch.empty_like(q)
    return _decode_append(_lib.ga_decode_global_hd512_append, "ga_decode_global_hd512_append",
                          k_new, v_new, q, k_pool, v_pool, page_table, seq_lens, window=None,
                          scale=scale, plan=plan, workspace=workspace, out=out, k_scale=k_scale,
                          v_scale=v_scale, err_word=err_word, stream=stream)


NOALLOC_SCRATCH_BYTES = 64 << 20


def ga_decode_global_hd512_noalloc(q, k_pool, v_pool, page_table, seq_lens, *, scale, plan,
                                   out, k_scale=None, v_scale=None, err_word=None, stream=None):
    """Global decode whose split-KV scratch is the library's built-in device
    array (no workspace argument): for callers that cannot allocate device
    memory at decode time.  Calls that overlap on the GPU share that array and
    race; plans needing more than NOALLOC_SCRATCH_BYTES are rejected."""
    B, Hq = q.shape[0], q.shape[1]
    st = _lib.ga_decode_global_hd512_noalloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _kv_dtype(k_pool), _ptr(k_scale), _ptr(v_scale),
        _ptr(page_table), page_table.shape[1], _ptr(seq_lens), B, Hq, k_pool.shape[1],
        k_pool.shape[2], k_pool.shape[0], float(scale), ctypes.byref(plan), _ptr(out),
        _ptr(err_word), _stream(stream))
    _check(st, "ga_decode_global_hd512_noalloc")
    return out


def ga_splitkv_combine(partial_o, partial_lse, plan, seq_lens, pt_stride, out, *, err_word=None,
                       stream=None):
    st = _lib.ga_splitkv_combine(_ptr(partial_o), _ptr(partial_lse), ctypes.byref(plan),
                                 _ptr(seq_lens), int(pt_stride), _ptr(out), _ptr(err_word),
                                 _stream(stream))
    _check(st, "ga_splitkv_combine")
    return out


def ga_check_error_word(word: int) -> int:
    return int(_lib.ga_check_error_word(int(word)))


def ga_read_stream(src: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """One read of every byte of src (measurement helper: the HBM read
    ceiling); sink is a device int64 tensor of one element."""
    _check(_lib.ga_read_stream(_ptr(src), src.numel() * src.element_size(), _ptr(sink),
                               _stream(stream)), "ga_read_stream")


def workspace_views(plan: ga_plan, workspace: torch.Tensor):
    """(partial_o [rc, Hq * S, D], partial_lse [rc, Hq * S], touch_log [rc, stride]) views
    (S = plan.q_len; column h * S + i is query i of head h)."""
    rc, Hq, D = plan.row_chunks, plan.num_q_heads * plan.q_len, plan.head_dim
    po = plo = log = None
    if plan.mode != GA_SPLIT_NONE:
        po = workspace[plan.partial_o_offset: plan.partial_o_offset + rc * Hq * D * 4] \
            .view(torch.float32).view(rc, Hq, D)
        plo = workspace[plan.partial_lse_offset: plan.partial_lse_offset + rc * Hq * 4] \
            .view(torch.float32).view(rc, Hq)
    if plan.flags & GA_PLAN_TOUCH_LOG:
        n = rc * plan.touch_stride
        log = workspace[plan.touch_log_offset: plan.touch_log_offset + n * 4] \
            .view(torch.int32).view(rc, plan.touch_stride)
    return po, plo, log


def ga_plan_splits_mq(seq_lens_host: Sequence[int], *, q_len: int, **kw) -> ga_plan:
    """Multi-query planner: q_len query tokens per row (the last q_len positions)."""
    return ga_plan_splits(seq_lens_host, q_len=q_len, **kw)
