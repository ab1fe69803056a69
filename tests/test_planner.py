"""Host-side split-KV planner (no GPU): modes, capacity, workspace layout,
SM filling and the chunk rule that keeps rows batch-invariant."""
import numpy as np
import pytest

from paged_split_kv_gqa_gb300 import workloads as W


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _pages(L, Wn):
    lo = max(0, L - Wn) if Wn > 0 else 0
    return 0 if L == 0 else (L - 1) // 16 - lo // 16 + 1


def test_no_split(ga):
    p = ga.ga_plan_splits([40, 33], num_q_heads=4, num_kv_heads=2, head_dim=256, window=32,
                          num_sms=152, requested_splits=1)
    assert p.mode == ga.GA_SPLIT_NONE and p.workspace_bytes == 0
    assert p.row_chunks == 2 and p.units == 4 and p.grid == 4


@pytest.mark.parametrize("s", [2, 4, 8, 16])
def test_fixed_count(ga, s):
    lens = [40, 33, 1, 0, 1025]
    p = ga.ga_plan_splits(lens, num_q_heads=8, num_kv_heads=2, head_dim=512, window=0,
                          num_sms=152, requested_splits=s)
    assert p.mode == ga.GA_SPLIT_COUNT and p.splits == s
    rc = 0
    for L in lens:
        n = _pages(L, 0)
        cp = -(-n // s) if n else 1
        rc += -(-n // cp) if n else 1
    assert p.row_chunks == rc
    assert p.workspace_bytes >= rc * 8 * 512 * 4 + rc * 8 * 4
    assert p.partial_lse_offset >= p.partial_o_offset + rc * 8 * 512 * 4
    assert p.partial_o_offset % 256 == 0 and p.partial_lse_offset % 256 == 0


def test_fixed_chunk_is_per_row(ga):
    lens = [4096, 100, 17]
    p = ga.ga_plan_splits(lens, num_q_heads=32, num_kv_heads=4, head_dim=512, window=0,
                          num_sms=152, fixed_chunk_tokens=512)
    assert p.mode == ga.GA_SPLIT_CHUNK and p.chunk_pages == 32
    assert p.row_chunks == 8 + 1 + 1
    # a row's chunk count depends only on its own length
    q = ga.ga_plan_splits([4096], num_q_heads=32, num_kv_heads=4, head_dim=512, window=0,
                          num_sms=152, fixed_chunk_tokens=512)
    assert q.row_chunks == 8


def test_touch_log_capacity(ga):
    p = ga.ga_plan_splits([40, 33, 300], num_q_heads=4, num_kv_heads=2, head_dim=256, window=32,
                          num_sms=8, requested_splits=1, flags=ga.GA_PLAN_TOUCH_LOG)
    assert p.touch_stride == 3 and p.workspace_bytes >= 3 * 3 * 4


def test_auto_fills_sms_for_long_context(ga):
    wl = W.config(4)
    p = ga.ga_plan_splits(wl.seq_lens, num_q_heads=32, num_kv_heads=4, head_dim=512, window=0,
                          num_sms=152)
    assert p.mode == ga.GA_SPLIT_CHUNK
    assert p.units >= 152 and p.grid == 152


def test_auto_31b_global_splits_uneven_rows(ga):
    wl = W.config(3)
    p = ga.ga_plan_splits(wl.seq_lens, num_q_heads=32, num_kv_heads=4, head_dim=512, window=0,
                          num_sms=152)
    assert p.mode == ga.GA_SPLIT_CHUNK and p.units >= 4 * 152


def test_auto_local_window_big_batch(ga):
    wl = W.config(3)
    p = ga.ga_plan_splits(wl.seq_lens, num_q_heads=32, num_kv_heads=16, head_dim=256, window=1024,
                          num_sms=152)
    # 1024 units of 65 pages each already fill 152 SMs well
    assert p.units >= 1024 and p.grid == 152


def test_invalid(ga):
    base = dict(num_q_heads=4, num_kv_heads=2, head_dim=256, window=32, num_sms=8)
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits([40], **dict(base, head_dim=128))
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits([40], **dict(base, page_size=32))
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits([40], **base, requested_splits=2, fixed_chunk_tokens=32)
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits([40], **base, fixed_chunk_tokens=24)
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits([-1], **base)
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits(np.ones(4097, dtype=np.int32), **base)
    p = ga.ga_plan_splits([], **base)
    assert p.units == 0 and p.grid == 1
