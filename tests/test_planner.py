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


def _chunks(L, Wn, mode, s=0, cp=0):
    n = _pages(L, Wn)
    if n == 0 or mode == "none":
        return 1
    per = -(-n // s) if mode == "count" else cp
    return -(-n // per)


@pytest.mark.parametrize("seed", range(12))
def test_multi_query_plan_properties(ga, seed):
    """Seeded random multi-query plans: the column tile follows the unit rule
    (8 up to 8 columns per kv head; 64 from 32 columns at hd512 / 64 at hd256 or
    when tensor-core units are asked for; else 32), and units, grid, row chunks
    (union window W + S - 1) and the partials' workspace follow from it."""
    rng = np.random.default_rng(500 + seed)
    D = int(rng.choice([256, 512]))
    Hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 3, 8]))
    S = int(rng.choice([1, 2, 4, 5, 8, 16, 33, 64]))
    Wn = int(rng.choice([0, 32, 1024])) if D == 256 else 0
    lens = [int(x) for x in rng.integers(0, 3000, size=int(rng.integers(1, 12)))]
    flags = int(rng.choice([0, ga.GA_PLAN_TENSOR_CORE_UNITS, ga.GA_PLAN_COLUMN_PARALLEL_UNITS]))
    split = [dict(requested_splits=1), dict(requested_splits=3), dict(fixed_chunk_tokens=64)][
        seed % 3]
    p = ga.ga_plan_splits_mq(lens, q_len=S, num_q_heads=g * Hkv, num_kv_heads=Hkv, head_dim=D,
                             window=Wn, num_sms=152, flags=flags, **split)
    cols = g * S
    if cols <= 8:
        tile = 8
    elif flags == ga.GA_PLAN_TENSOR_CORE_UNITS:
        tile = 64
    elif flags == ga.GA_PLAN_COLUMN_PARALLEL_UNITS:
        tile = 32
    else:
        tile = 64 if cols >= (32 if D == 512 else 64) else 32
    assert p.col_tile == tile and p.q_len == S
    w_union = Wn + S - 1 if Wn else 0
    mode = "none" if "requested_splits" in split and split["requested_splits"] == 1 else \
        ("count" if "requested_splits" in split else "chunk")
    rc = sum(_chunks(L, w_union, mode, s=split.get("requested_splits", 0),
                     cp=split.get("fixed_chunk_tokens", 0) // 16) for L in lens)
    assert p.row_chunks == rc
    assert p.units == rc * Hkv * -(-cols // tile)
    assert p.grid == max(1, min(p.units, 152))
    if p.mode != ga.GA_SPLIT_NONE:
        assert p.partial_lse_offset >= p.partial_o_offset + rc * g * Hkv * S * D * 4
        assert p.partial_o_offset % 256 == 0 and p.partial_lse_offset % 256 == 0
        assert p.workspace_bytes >= p.partial_lse_offset + rc * g * Hkv * S * 4


def test_units_span_several_kv_heads(ga):
    """With GA_PLAN_KV_E4M3 the planner gives the E4M3 sliding family units of
    8 / group kv heads only when the one-head plan needs no split and the wider
    units fill at least four rounds of the SMs; otherwise one kv head."""
    kw = dict(num_q_heads=32, num_kv_heads=16, head_dim=256, window=1024, num_sms=152)
    few = [3000] * 8                              # 32 four-head units: too few
    one = ga.ga_plan_splits(few, **kw)
    p = ga.ga_plan_splits(few, flags=ga.GA_PLAN_KV_E4M3, **kw)
    assert one.kv_heads_per_unit == 1 and p.kv_heads_per_unit == 1 and p.units == one.units
    many = W.config(5).seq_lens                   # 256 rows: 1024 four-head units
    p = ga.ga_plan_splits(many, flags=ga.GA_PLAN_KV_E4M3, **kw)
    assert p.mode == ga.GA_SPLIT_NONE and p.kv_heads_per_unit == 4 and p.units == 256 * 4
    assert ga.ga_plan_splits(many, **kw).kv_heads_per_unit == 1     # bf16 plan
    # group 4: two kv heads per unit; group 1: never
    p = ga.ga_plan_splits(many, flags=ga.GA_PLAN_KV_E4M3,
                          **dict(kw, num_q_heads=64))
    assert p.kv_heads_per_unit == 2 and p.units == 256 * 8
    p = ga.ga_plan_splits(many, flags=ga.GA_PLAN_KV_E4M3, **dict(kw, num_q_heads=16))
    assert p.kv_heads_per_unit == 1
    # the global family (head_dim 512) and multi-query plans keep one kv head
    assert ga.ga_plan_splits(many, flags=ga.GA_PLAN_KV_E4M3,
                             **dict(kw, head_dim=512, window=0)).kv_heads_per_unit == 1


def _snake(s, G, U):
    """Slot s of G CTAs over U units -> position in the sorted order: every
    odd pass over the CTAs runs backwards (the deal the header documents)."""
    r, q = divmod(s, G)
    n = min(G, U - r * G)
    return r * G + (n - 1 - q if r % 2 else q)


@pytest.mark.parametrize("G,U", [(152, 1024), (152, 152), (7, 50), (5, 3), (40, 512)])
def test_snake_deal_is_a_permutation(G, U):
    pos = [_snake(s, G, U) for s in range(U)]
    assert sorted(pos) == list(range(U))
    # CTA q takes slots q, q + G, ...: in a full odd pass it gets position G - 1 - q
    if U >= 2 * G:
        assert pos[G] == 2 * G - 1 and pos[2 * G - 1] == G


def test_rows_by_size_schedule(ga):
    """The planner deals one-chunk plans of unequal rows longest first (snake
    order) when that evens out the CTA loads; equal rows, split plans and
    multi-query plans keep round robin.  The choice is checked against the
    same deal simulated here: the busiest CTA's pages drop."""
    kw = dict(num_q_heads=32, num_kv_heads=16, head_dim=256, window=1024, num_sms=152)
    lens = W.config(5).seq_lens
    p = ga.ga_plan_splits(lens, flags=ga.GA_PLAN_KV_E4M3, **kw)
    assert p.mode == ga.GA_SPLIT_NONE and p.schedule == ga.GA_SCHEDULE_ROWS_BY_SIZE
    upr = 16 // p.kv_heads_per_unit
    pages = [_pages(int(L), 1024) for L in lens]
    order = sorted(range(len(lens)), key=lambda b: (-min(pages[b], 256), b))
    G, U = p.grid, p.units
    rr, sn = np.zeros(G), np.zeros(G)
    for s in range(U):
        rr[s % G] += pages[s // upr]
        sn[s % G] += pages[order[_snake(s, G, U) // upr]]
    assert rr.sum() == sn.sum() and sn.max() < 0.97 * rr.max()
    # equal rows: nothing to gain
    q = ga.ga_plan_splits([20000] * 64, **kw)
    assert q.mode == ga.GA_SPLIT_NONE and q.schedule == ga.GA_SCHEDULE_ROUND_ROBIN
    # split plans and multi-query plans: round robin
    assert ga.ga_plan_splits(lens, requested_splits=2, **kw).schedule == 0
    assert ga.ga_plan_splits_mq(lens, q_len=4, **kw).schedule == 0
    # the row order and its counters must fit after the row prefix
    big = np.random.default_rng(0).integers(1, 3000, 1792)
    assert ga.ga_plan_splits(big, requested_splits=1, **kw).schedule == 0


def test_e4m3_unit_cost(ga):
    """E4M3 plans weigh a unit's fixed cost (the tcgen05 kernel's start and
    drain) at 18 pages: the ragged batch's first 4 rows stay unsplit for the
    E4M3 sliding family (measured faster: 15.6 against 19.2 us a layer with
    16-page chunks), while the same rows as a bf16 plan, whose units cost 4
    pages, are chunked; one row is chunked either way."""
    kw = dict(num_q_heads=32, num_kv_heads=16, head_dim=256, window=1024, num_sms=152)
    lens = W.config(5).seq_lens
    assert ga.ga_plan_splits(lens[:4], flags=ga.GA_PLAN_KV_E4M3, **kw).mode == ga.GA_SPLIT_NONE
    assert ga.ga_plan_splits(lens[:4], **kw).mode == ga.GA_SPLIT_CHUNK
    assert ga.ga_plan_splits(lens[:1], flags=ga.GA_PLAN_KV_E4M3, **kw).mode == ga.GA_SPLIT_CHUNK


@pytest.mark.parametrize("Hq,Hkv,D,W_,S,tile", [
    (16, 2, 512, 0, 1, 8),        # 8 columns per kv head
    (16, 2, 512, 0, 2, 16),       # 16
    (16, 2, 512, 0, 3, 16),       # 24: two units, the second half full
    (16, 2, 512, 0, 4, 16),       # 32
    (32, 2, 512, 0, 1, 16),       # a GQA group of 16 at one query
    (8, 4, 256, 1024, 4, 8),      # 8
    (8, 4, 256, 1024, 8, 16),     # 16
    (8, 2, 256, 32, 3, 16),       # 12: one unit with 4 idle columns
])
def test_e4m3_plans_ask_for_16_column_units(ga, Hq, Hkv, D, W_, S, tile):
    """A plan made with GA_PLAN_KV_E4M3 for more than 8 (query, head) columns
    per kv head asks the E4M3 kernel for units of 16 columns and counts its
    units so; the same shape without the flag keeps the bf16 tiles."""
    lens = [0, 1, 17, 300, 2049, 40]
    kw = dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, window=W_, num_sms=152,
              requested_splits=2)
    p = ga.ga_plan_splits(lens, flags=ga.GA_PLAN_KV_E4M3, q_len=S, **kw)
    cols = Hq // Hkv * S
    assert p.col_tile == tile and p.kv_heads_per_unit == 1
    assert p.units == p.row_chunks * Hkv * -(-cols // tile)
    plain = ga.ga_plan_splits(lens, q_len=S, **kw)
    assert plain.col_tile != 16 and plain.row_chunks == p.row_chunks


def _chunk_deal_load(lens, cp, Hkv, G, sort):
    """Pages per CTA of a chunked plan under round robin or the rows-by-size
    deal as the header documents it: the full chunks in row order, then the
    rows' shorter last chunks longest first (ties in row order), dealt in
    snake order."""
    rc_sizes = []                                  # row-chunks in row order
    for L in lens:
        n = _pages(int(L), 0)
        rc_sizes += [min(cp, n - j * cp) for j in range(-(-n // cp))] if n else [0]
    full = [s for s in rc_sizes if s == cp]
    last = sorted((s for s in rc_sizes if s != cp), key=lambda s: -min(s, 256))
    order = full + last if sort else rc_sizes
    U = len(order) * Hkv
    load = np.zeros(G)
    for s in range(U):
        load[s % G] += order[(_snake(s, G, U) if sort else s) // Hkv]
    return load


def test_rows_by_size_deal_of_chunked_plans(ga):
    """Plans in fixed-size chunks take the rows-by-size deal too (full chunks
    first, then the shorter last chunks longest first) when it evens the CTA
    loads out: the 31B global family's chunked plans (bf16 and E4M3 pools)
    and the ragged batch's; the busiest CTA's pages drop as simulated here.
    Split-count plans and batches above 596 rows keep round robin."""
    for idx, flags in ((3, 0), (3, "e4m3"), (5, 0)):
        wl = W.config(idx)
        fam = wl.global_
        p = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                              num_kv_heads=fam.num_kv_heads, head_dim=512, window=0,
                              num_sms=152, flags=ga.GA_PLAN_KV_E4M3 if flags else 0)
        assert p.mode == ga.GA_SPLIT_CHUNK and p.schedule == ga.GA_SCHEDULE_ROWS_BY_SIZE
        rr = _chunk_deal_load(wl.seq_lens, p.chunk_pages, fam.num_kv_heads, p.grid, False)
        sn = _chunk_deal_load(wl.seq_lens, p.chunk_pages, fam.num_kv_heads, p.grid, True)
        assert rr.sum() == sn.sum() and sn.max() < 0.97 * rr.max(), (idx, flags)
    lens = W.config(3).seq_lens
    kw = dict(num_q_heads=32, num_kv_heads=4, head_dim=512, window=0, num_sms=152)
    assert ga.ga_plan_splits(lens, requested_splits=4, **kw).schedule == 0
    big = np.random.default_rng(1).integers(8000, 30000, 597)
    assert ga.ga_plan_splits(big, fixed_chunk_tokens=2048, **kw).schedule == 0
