"""The rows-by-size deal of work units (GA_SCHEDULE_ROWS_BY_SIZE: rows in
descending order of attended pages, or for a plan in fixed-size chunks the
full chunks first and the rows' shorter last chunks longest first; every
other pass over the CTAs reversed) changes which CTA takes a unit, never
what a unit computes: every
decode kernel's outputs are bit-identical to the round-robin deal, the page
sets read are the same, the fused append writes the same pools, and sampled
rows match the oracle.  Batches with more units than CTAs (the plan made
for 40 SMs) and unequal rows, including empty ones.  ("[Model] Gemma 4 M3
31B", Proposed Plan: the split-KV / work policy re-checked per geometry.)"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode_rows_gathered, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"
_rng = np.random.default_rng(11)
LENS = [int(x) for x in np.clip(np.exp(_rng.normal(6.5, 1.2, 96)), 0, 4000).astype(int)]
LENS[:6] = [0, 1, 16, 1023, 1024, 1025]

CASES = {
    "local_bf16": (W.Family("local", 16, 8, 256, 1024), {}),
    "local_e4m3": (W.Family("local", 16, 8, 256, 1024, 1), {}),
    "local_e4m3_4_heads": (W.Family("local", 16, 8, 256, 1024, 1), {"heads": 4}),
    "local_e4m3_kv_alias": (W.Family("local", 16, 8, 256, 1024, 1), {"alias": True}),
    "global_bf16_unsplit": (W.Family("global", 16, 2, 512, 0), {}),
    "global_e4m3_unsplit": (W.Family("global", 16, 2, 512, 0, 1), {}),
    "global_bf16_chunked": (W.Family("global", 16, 2, 512, 0), {"chunk": 128}),
    "global_e4m3_chunked": (W.Family("global", 16, 2, 512, 0, 1), {"chunk": 256}),
    "local_bf16_chunked": (W.Family("local", 16, 8, 256, 1024), {"chunk": 208}),
    "global_e4m3_chunked_16_columns": (W.Family("global", 32, 2, 512, 0, 1), {"chunk": 96}),
}


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _setup(case):
    fam, opt = CASES[case]
    wl = W.Workload("schedule", np.asarray(LENS, dtype=np.int32), 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=23, poison=True,
                              release_old=fam.window > 0)
    if opt.get("alias"):
        fi = dataclasses.replace(fi, v_pool=fi.k_pool, v_scale=fi.k_scale)
    return fam, opt, fi


def _plans(ga, fam, opt, flags=0):
    kw = dict(num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
              head_dim=fam.head_dim, window=fam.window, num_sms=40,
              flags=flags | (ga.GA_PLAN_KV_E4M3 if fam.kv_dtype == W.KV_E4M3 else 0))
    if "chunk" in opt:
        kw["fixed_chunk_tokens"] = opt["chunk"]
    else:
        kw["requested_splits"] = 1
    out = []
    for sched in (ga.GA_SCHEDULE_ROUND_ROBIN, ga.GA_SCHEDULE_ROWS_BY_SIZE):
        plan = ga.ga_plan_splits(LENS, **kw)
        if opt.get("heads"):
            plan.kv_heads_per_unit = opt["heads"]
        plan.schedule = sched
        assert plan.units > plan.grid
        out.append(plan)
    return out


def _bits(t):
    return t.contiguous().view(torch.uint8)


@pytest.mark.parametrize("case", sorted(CASES))
def test_deal_changes_no_bit(ga, case):
    fam, opt, fi = _setup(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for plan in _plans(ga, fam, opt):
        outs.append(run_decode(ga, fi, plan, err=err, out=torch.full_like(fi.q, float("nan"))))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(outs[0]), _bits(outs[1])), case
    rows = sorted(set([0, 1, 3, 4, 5] + W.sample_rows(len(LENS), 6, seed=2).tolist()))
    assert_close(outs[1][rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=fam.kv_dtype, what=case)


@pytest.mark.parametrize("case", ["local_bf16", "local_e4m3_4_heads", "local_bf16_chunked"])
def test_deal_reads_the_same_pages(ga, case):
    """Touch log (one entry list per row-chunk): the same physical pages per
    row-chunk under both deals, and per row (its chunks in order) equal to
    the oracle's window pages."""
    fam, opt, fi = _setup(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    logs = []
    for plan in _plans(ga, fam, opt, flags=ga.GA_PLAN_TOUCH_LOG):
        if opt.get("heads"):
            plan.kv_heads_per_unit = opt["heads"]
        ws = ga.workspace_for(plan, DEV)
        _, _, log = ga.workspace_views(plan, ws)
        log.fill_(-1)
        run_decode(ga, fi, plan, err=err, workspace=ws)
        torch.cuda.synchronize()
        logs.append(log.cpu().numpy().copy())
    assert int(err.item()) == 0
    assert np.array_equal(logs[0], logs[1])
    table = fi.page_table.cpu().numpy()
    cp = opt.get("chunk", 0) // 16
    rc = 0
    for b, L in enumerate(LENS):
        first, n = O.logical_pages(L, fam.window, 16)
        chunks = max(1, -(-n // cp)) if cp else 1
        got = [int(x) for r in range(rc, rc + chunks) for x in logs[1][r] if x >= 0]
        rc += chunks
        assert got == [int(table[b, p]) for p in range(first, first + n)], (b, L)


@pytest.mark.parametrize("case", ["local_bf16", "local_e4m3", "local_e4m3_4_heads",
                                  "local_bf16_chunked"])
def test_deal_with_fused_append(ga, case):
    """The decode call with the append fused in: same pools and outputs under
    both deals (the unit that holds a row's last page writes its token)."""
    fam, opt, fi = _setup(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = []
    for plan in _plans(ga, fam, opt):
        k, v = fi.k_pool.clone(), fi.v_pool.clone()
        out = torch.empty_like(fi.q)
        ga.ga_decode_local_hd256_append(fi.k_new, fi.v_new, fi.q, k, v, fi.page_table,
                                        fi.seq_lens, window=fam.window,
                                        scale=1 / math.sqrt(fam.head_dim), plan=plan,
                                        workspace=ga.workspace_for(plan, DEV), out=out,
                                        k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
        torch.cuda.synchronize()
        res.append((k, v, out))
    assert int(err.item()) == 0
    for a, b in zip(res[0], res[1]):
        assert torch.equal(_bits(a), _bits(b)), case


def test_ragged_batch_deal_sampled(ga):
    """The ragged 256-row batch in the bench's launch configuration: the
    planner deals rows by size, and sampled rows match the oracle."""
    wl = W.config(5)
    fam = wl.local
    fi = W.make_family_inputs(wl, fam, device=DEV, poison=True, release_old=True, seed=3)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=256, window=fam.window,
                             flags=ga.GA_PLAN_KV_E4M3)
    assert plan.schedule == ga.GA_SCHEDULE_ROWS_BY_SIZE and plan.kv_heads_per_unit == 4
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_decode(ga, fi, plan, err=err)
    plan0 = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                              num_kv_heads=fam.num_kv_heads, head_dim=256, window=fam.window,
                              flags=ga.GA_PLAN_KV_E4M3)
    plan0.schedule = ga.GA_SCHEDULE_ROUND_ROBIN
    out0 = run_decode(ga, fi, plan0, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(out), _bits(out0))
    rows = W.sample_rows(wl.batch, 12, seed=4)
    assert_close(out[rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=1, what="ragged rows-by-size")


def test_deal_at_the_batch_limit(ga):
    """1791 rows, the most the rows-by-size deal takes (its row order and
    counters fill the row-prefix array exactly): bit-identical to round robin
    and sampled rows against the oracle; 1792 rows with the deal forced are
    refused before any launch."""
    fam = W.Family("local", 2, 1, 256, 64)
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 200, 1791)]
    wl = W.Workload("limit", np.asarray(lens, dtype=np.int32), 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=9, poison=True, release_old=True)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for sched in (ga.GA_SCHEDULE_ROUND_ROBIN, ga.GA_SCHEDULE_ROWS_BY_SIZE):
        plan = ga.ga_plan_splits(lens, num_q_heads=2, num_kv_heads=1, head_dim=256, window=64,
                                 requested_splits=1, num_sms=40)
        plan.schedule = sched
        outs.append(run_decode(ga, fi, plan, err=err, out=torch.full_like(fi.q, float("nan"))))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(_bits(outs[0]), _bits(outs[1]))
    rows = W.sample_rows(len(lens), 10, seed=6)
    assert_close(outs[1][rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=0, what="1791 rows")
    lens2 = lens + [5]
    wl2 = W.Workload("limit+1", np.asarray(lens2, dtype=np.int32), 16, fam, fam)
    fi2 = W.make_family_inputs(wl2, fam, device=DEV, seed=9, release_old=True)
    plan = ga.ga_plan_splits(lens2, num_q_heads=2, num_kv_heads=1, head_dim=256, window=64,
                             requested_splits=1, num_sms=40)
    plan.schedule = ga.GA_SCHEDULE_ROWS_BY_SIZE
    with pytest.raises(ga.GAError) as exc:
        run_decode(ga, fi2, plan, err=err)
    assert exc.value.status == ga.GA_ERR_INVALID_ARG


def test_chunked_deal_limits(ga):
    """A chunked plan takes the deal up to 596 rows (its three sorted arrays
    and counters fill the row-prefix array); 597 rows, or a plan split into a
    fixed number of chunks per row, with the deal forced are refused before
    any launch."""
    fam = W.Family("global", 2, 1, 512, 0)
    rng = np.random.default_rng(8)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for n, ok in ((596, True), (597, False)):
        lens = [int(x) for x in rng.integers(0, 300, n)]
        wl = W.Workload("climit", np.asarray(lens, dtype=np.int32), 16, fam, fam)
        fi = W.make_family_inputs(wl, fam, device=DEV, seed=4)
        outs = []
        for sched in (ga.GA_SCHEDULE_ROUND_ROBIN, ga.GA_SCHEDULE_ROWS_BY_SIZE):
            plan = ga.ga_plan_splits(lens, num_q_heads=2, num_kv_heads=1, head_dim=512,
                                     window=0, fixed_chunk_tokens=64, num_sms=40)
            plan.schedule = sched
            if sched == ga.GA_SCHEDULE_ROWS_BY_SIZE and not ok:
                with pytest.raises(ga.GAError) as exc:
                    run_decode(ga, fi, plan, err=err)
                assert exc.value.status == ga.GA_ERR_INVALID_ARG
                continue
            outs.append(run_decode(ga, fi, plan, err=err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        if ok:
            assert torch.equal(_bits(outs[0]), _bits(outs[1]))
            rows = W.sample_rows(n, 6, seed=1)
            assert_close(outs[1][rows].float().cpu().numpy(),
                         oracle_decode_rows_gathered(fi, rows), what="596 rows, chunked deal")
    lens = [40, 300, 900, 17]
    wl = W.Workload("count", np.asarray(lens, dtype=np.int32), 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=4)
    plan = ga.ga_plan_splits(lens, num_q_heads=2, num_kv_heads=1, head_dim=512, window=0,
                             requested_splits=3)
    plan.schedule = ga.GA_SCHEDULE_ROWS_BY_SIZE
    with pytest.raises(ga.GAError) as exc:
        run_decode(ga, fi, plan, err=err)
    assert exc.value.status == ga.GA_ERR_INVALID_ARG
