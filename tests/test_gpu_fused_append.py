"""A decode step with the KV page append fused into the decode launch
(ga_decode_local_hd256_append, ga_decode_global_hd512_append): the unit that
reads a row's last page first writes the row's new token into it.  The pools
after the call and its outputs must be bit-identical to ga_kv_append (at
positions seq_lens - 1) followed by the plain decode, for every decode kernel
(bf16 page-parallel at both head dims, K == V, E4M3 on tcgen05 with one and
with four kv heads per unit, the E4M3 global family, its 16-column units at a
GQA group of 16), split or not, with empty rows; more than 8 query heads per
kv head on bf16 pools takes the two-launch path, same bits; K == V pools (one pool: the value token is the one that stays, as with
ga_kv_append); an invalid page at the token's slot is reported as by
ga_kv_append.
("[Model] Gemma 4 M1 12B", Description: paged decode, the step's token
appended at position L - 1 and attended.)"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [1500, 1024, 1025, 40, 16, 17, 0, 2222, 1]

CASES = {
    "local_bf16": (W.Family("local", 16, 8, 256, 1024), {}),
    "global_bf16": (W.Family("global", 16, 2, 512, 0), {}),
    "global_bf16_kv_alias": (W.Family("global", 16, 2, 512, 0), {"alias": True}),
    "local_e4m3": (W.Family("local", 16, 8, 256, 1024, 1), {}),
    "local_e4m3_4_heads": (W.Family("local", 16, 8, 256, 1024, 1), {"heads": 4}),
    "global_e4m3": (W.Family("global", 16, 2, 512, 0, 1), {}),
    "global_bf16_group16": (W.Family("global", 32, 2, 512, 0), {}),   # two-launch path
    "global_e4m3_group16": (W.Family("global", 32, 2, 512, 0, 1), {}),  # 16-column units
    "local_e4m3_2_heads": (W.Family("local", 16, 4, 256, 1024, 1), {"heads": 2}),
    "local_e4m3_kv_alias": (W.Family("local", 16, 8, 256, 1024, 1), {"alias": True}),
    "global_e4m3_kv_alias": (W.Family("global", 16, 2, 512, 0, 1), {"alias": True}),
}


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _setup(case, seed=41):
    fam, opt = CASES[case]
    wl = W.Workload("append", np.asarray(LENS, dtype=np.int32), 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=seed, poison=True,
                              release_old=fam.window > 0)
    if opt.get("alias"):
        fi = dataclasses.replace(fi, v_pool=fi.k_pool, v_scale=fi.k_scale)
    return fam, opt, fi


def _plan(ga, fam, opt, split):
    flags = ga.GA_PLAN_KV_E4M3 if fam.kv_dtype == W.KV_E4M3 else 0
    plan = ga.ga_plan_splits(LENS, num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
                             head_dim=fam.head_dim, window=fam.window, flags=flags, **split)
    if opt.get("heads"):
        plan.kv_heads_per_unit = opt["heads"]
    return plan


def _pools(fi):
    k = fi.k_pool.clone()
    v = k if fi.v_pool.data_ptr() == fi.k_pool.data_ptr() else fi.v_pool.clone()
    return k, v


def _bits(t):
    """Raw bytes (NaN poison compares equal to itself)."""
    return t.contiguous().view(torch.uint8)


def _same(a, b):
    return a.shape == b.shape and torch.equal(_bits(a), _bits(b))


def _kw(fam, fi, plan, ws, out, err, k_pool, v_pool):
    kw = dict(scale=1.0 / math.sqrt(fam.head_dim), plan=plan, workspace=ws, out=out,
              k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    if fam.window:
        kw["window"] = fam.window
    return kw


@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=3)],
                         ids=["s1", "s3"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_append_equals_append_then_decode(ga, case, split):
    fam, opt, fi = _setup(case)
    plan = _plan(ga, fam, opt, split)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # two-launch reference: ga_kv_append at L - 1, then the plain decode
    k1, v1 = _pools(fi)
    pos = (fi.seq_lens - 1).to(torch.int32)
    ga.ga_kv_append(fi.k_new, fi.v_new, k1, v1, fi.page_table, pos, k_scale=fi.k_scale,
                    v_scale=fi.v_scale, err_word=err)
    out1 = torch.full_like(fi.q, float("nan"))
    kw = _kw(fam, fi, plan, ga.workspace_for(plan, DEV), out1, err, k1, v1)
    dec = ga.ga_decode_local_hd256 if fam.window else ga.ga_decode_global_hd512
    dec(fi.q, k1, v1, fi.page_table, fi.seq_lens, **kw)
    # one call
    k2, v2 = _pools(fi)
    out2 = torch.full_like(fi.q, float("nan"))
    kw = _kw(fam, fi, plan, ga.workspace_for(plan, DEV), out2, err, k2, v2)
    fused = ga.ga_decode_local_hd256_append if fam.window else ga.ga_decode_global_hd512_append
    fused(fi.k_new, fi.v_new, fi.q, k2, v2, fi.page_table, fi.seq_lens, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same(k1, k2) and _same(v1, v2), f"{case}: pools differ"
    assert _same(out1, out2), f"{case}: outputs differ"
    # and against the oracle on the appended pools
    ref = oracle_decode(dataclasses.replace(fi, k_pool=k2, v_pool=v2))
    assert_close(out2.float().cpu().numpy(), ref, kv_dtype=fam.kv_dtype, what=case)


def test_fused_append_reports_bad_page(ga):
    """The page holding a row's token is invalid: GA_DEVERR_POSITION, as
    ga_kv_append reports it; no pool page changes for that row."""
    fam, opt, fi = _setup("local_bf16")
    plan = _plan(ga, fam, opt, dict(requested_splits=1))
    table = fi.page_table.clone()
    table[0, (LENS[0] - 1) // 16] = fi.num_pages + 3     # row 0's last page
    k2, v2 = _pools(fi)
    before = k2.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = _kw(fam, fi, plan, ga.workspace_for(plan, DEV), torch.empty_like(fi.q), err, k2, v2)
    ga.ga_decode_local_hd256_append(fi.k_new, fi.v_new, fi.q, k2, v2, table, fi.seq_lens, **kw)
    torch.cuda.synchronize()
    word = int(err.item())
    assert word & ga.GA_DEVERR_POSITION
    # the other rows' tokens were written
    for b, L in enumerate(LENS):
        if b == 0 or L == 0:
            continue
        page = int(table[b, (L - 1) // 16])
        assert _same(k2[page, :, (L - 1) % 16], fi.k_new[b]), b
    changed = (_bits(k2) != _bits(before)).flatten(1).any(dim=1)
    assert int(changed.sum()) == sum(1 for b, L in enumerate(LENS) if b != 0 and L > 0)


def test_fused_append_rejects_multi_query_plan(ga):
    fam, opt, fi = _setup("global_bf16")
    plan = ga.ga_plan_splits_mq(LENS, q_len=2, num_q_heads=16, num_kv_heads=2, head_dim=512,
                                window=0)
    with pytest.raises(ga.GAError) as exc:
        ga.ga_decode_global_hd512_append(fi.k_new, fi.v_new, fi.q, fi.k_pool, fi.v_pool,
                                         fi.page_table, fi.seq_lens, scale=0.1, plan=plan)
    assert exc.value.status == ga.GA_ERR_INVALID_ARG


FULL = {
    # (workload index, family, plan flags): the launch configurations the bench times
    "31b_local_bf16": (3, "local", 0),
    "31b_global_bf16": (3, "global", 0),
    "ragged_local_e4m3": (5, "local", "e4m3"),
    "ragged_global_bf16": (5, "global", 0),
}


@pytest.mark.parametrize("case", sorted(FULL))
def test_fused_append_full_size(ga, case):
    """Full-size batches with the bench's plans (several units per CTA, so the
    tcgen05 kernel's q warp writes the tokens of a CTA's later units): pools
    and outputs bit-identical to the two-launch step, and sampled rows
    against the oracle."""
    from tests.helpers import oracle_decode_rows_gathered
    idx, which, flags = FULL[case]
    wl = W.config(idx)
    fam = wl.local if which == "local" else wl.global_
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=5, poison=True,
                              release_old=fam.window > 0)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window,
                             flags=ga.GA_PLAN_KV_E4M3 if flags == "e4m3" else 0)
    if case == "ragged_local_e4m3":
        assert plan.kv_heads_per_unit == 4
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = ga.workspace_for(plan, DEV)
    k1, v1 = _pools(fi)
    pos = (fi.seq_lens - 1).to(torch.int32)
    ga.ga_kv_append(fi.k_new, fi.v_new, k1, v1, fi.page_table, pos, k_scale=fi.k_scale,
                    v_scale=fi.v_scale, err_word=err)
    out1 = torch.empty_like(fi.q)
    dec = ga.ga_decode_local_hd256 if fam.window else ga.ga_decode_global_hd512
    dec(fi.q, k1, v1, fi.page_table, fi.seq_lens, **_kw(fam, fi, plan, ws, out1, err, k1, v1))
    k2, v2 = fi.k_pool, fi.v_pool            # appended in place by the fused call
    out2 = torch.empty_like(fi.q)
    fused = ga.ga_decode_local_hd256_append if fam.window else ga.ga_decode_global_hd512_append
    fused(fi.k_new, fi.v_new, fi.q, k2, v2, fi.page_table, fi.seq_lens,
          **_kw(fam, fi, plan, ws, out2, err, k2, v2))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _same(out1, out2), f"{case}: outputs differ"
    assert _same(k1, k2) and _same(v1, v2), f"{case}: pools differ"
    del k1, v1
    rows = W.sample_rows(wl.batch, 8)
    assert_close(out2[rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=fam.kv_dtype, what=case)
    del fi
    torch.cuda.empty_cache()
