"""The sliding family's E4M3 decode with units of several kv heads (plans made
with GA_PLAN_KV_E4M3: 4 kv heads per unit at GQA group 2, 2 at group 4), whose
producer copies a page's blocks of those heads as one box per 128-dim region.
Checked against the fp64 oracle on the stored codes (3e-2 / 1.5e-2) over the
window edges 1023 / 1024 / 1025, short and empty rows and every split mode;
per-head NaN isolation (a NaN in one kv head's attended K or V reaches that
head's query heads only, as in the definition); the page set read, bit-exact;
and the full-size 31B-shaped batch on sampled rows.  ("[Model] Gemma 4 M2
26B-A4B", Proposed Plan: opt-in FP8 pool for the sliding family; "[Model]
Gemma 4 M3 31B", Acceptance Criteria: the 1023 / 1024 / 1025 window
boundaries.)"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import (assert_close, oracle_decode, oracle_decode_rows_gathered,
                           run_decode)

pytestmark = pytest.mark.gpu
DEV = "cuda"
LENS = [1023, 1024, 1025, 40, 2500, 1, 0, 17, 1600, 16]
SPLITS = [dict(requested_splits=1), dict(requested_splits=3), dict(fixed_chunk_tokens=48),
          dict()]


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


@pytest.fixture
def err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _inputs(lens, fam, seed, **kw):
    wl = W.Workload("heads", np.asarray(lens, dtype=np.int32), 16, fam, fam)
    kw.setdefault("poison", True)
    return W.make_family_inputs(wl, fam, device=DEV, seed=seed, **kw)


def _plan(ga, fi, flags=0, **kw):
    """A plan for E4M3 pools with units of 8 / group kv heads set explicitly
    (the planner picks them only for large batches)."""
    fam = fi.family
    plan = ga.ga_plan_splits(fi.seq_lens.cpu().numpy(), num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window, flags=ga.GA_PLAN_KV_E4M3 | flags, **kw)
    plan.kv_heads_per_unit = 8 // (fam.num_q_heads // fam.num_kv_heads)
    return plan


@pytest.mark.parametrize("split", SPLITS, ids=lambda s: str(s))
@pytest.mark.parametrize("Hq,Hkv,window", [(16, 8, 1024), (16, 4, 1024), (8, 4, 32),
                                           (32, 16, 1 << 20)])
def test_multi_head_units_vs_oracle(ga, err, Hq, Hkv, window, split):
    fam = W.Family("local", Hq, Hkv, 256, window, W.KV_E4M3)
    fi = _inputs(LENS, fam, seed=31, release_old=window < (1 << 20))
    plan = _plan(ga, fi, **split)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle_decode(fi)
    got = out.float().cpu().numpy()
    assert_close(got, ref, kv_dtype=1, what=f"Hq={Hq} Hkv={Hkv} W={window} {split}")
    assert np.all(got[np.asarray(LENS) == 0] == 0)


@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=3)])
def test_nan_stays_in_its_kv_head(ga, err, split):
    """A NaN in an attended K row of kv head 1 and one in an attended V row of
    kv head 2 (same unit of 4 heads) make only those heads' query heads NaN."""
    fam = W.Family("local", 16, 8, 256, 1024, W.KV_E4M3)
    fi = _inputs([100, 70, 1300], fam, seed=16, poison=False)
    p0 = int(fi.page_table[0, 3])                 # row 0, keys 48..63
    fi.k_pool[p0, 1, 5, 7] = W.E4M3_NAN_CODE      # kv head 1 -> query heads 2, 3
    p2 = int(fi.page_table[2, 40])                # row 2, keys 640..655 (in the window)
    fi.v_pool[p2, 2, 2, 100] = W.E4M3_NAN_CODE    # kv head 2 -> query heads 4, 5
    out = run_decode(ga, fi, _plan(ga, fi, **split), err=err).float().cpu().numpy()
    torch.cuda.synchronize()
    ref = oracle_decode(fi)
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    assert np.isnan(out[0, 2:4]).all() and np.isnan(out[2, 4:6, 100]).all()
    assert not np.isnan(out[0, :2]).any() and not np.isnan(out[0, 4:]).any()
    assert not np.isnan(out[2, :4]).any() and not np.isnan(out[2, 6:]).any()
    ok = ~np.isnan(ref)
    assert_close(out[ok], ref[ok], kv_dtype=1, what="finite part")


@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=4)])
def test_page_set_bit_exact(ga, err, split):
    lens = [40, 33, 1023, 1024, 1025, 2049, 3000, 1, 0]
    fam = W.Family("local", 16, 8, 256, 1024, W.KV_E4M3)
    fi = _inputs(lens, fam, seed=5, release_old=True)
    plan = _plan(ga, fi, flags=ga.GA_PLAN_TOUCH_LOG, **split)
    ws = ga.workspace_for(plan, DEV)
    _, _, log = ga.workspace_views(plan, ws)
    log.fill_(-1)
    run_decode(ga, fi, plan, err=err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    log = log.cpu().numpy()
    table = fi.page_table.cpu().numpy()
    rc = 0
    for b, L in enumerate(lens):
        first, n = O.logical_pages(L, fam.window, 16)
        want = [int(table[b, p]) for p in range(first, first + n)]
        got = []
        while True:
            got += [int(x) for x in log[rc] if x >= 0]
            rc += 1
            if n == 0 or len(got) >= len(want):
                break
        assert got == want, (b, L)
    assert rc == plan.row_chunks


@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=4), dict()],
                         ids=["s1", "s4", "auto"])
def test_31b_sampled(ga, err, split):
    wl = W.config(3)
    base = wl.local
    fam = W.Family("local", base.num_q_heads, base.num_kv_heads, 256, base.window, W.KV_E4M3)
    fi = W.make_family_inputs(wl, fam, device=DEV, poison=True, release_old=True)
    out = run_decode(ga, fi, _plan(ga, fi, **split), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 8)
    assert_close(out[rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=1, what=f"31B local E4M3 4-head units {split}")
    del fi
    torch.cuda.empty_cache()


def test_ragged_sampled(ga, err):
    """The ragged 256-row batch (lognormal lengths, E4M3 sliding family) in the
    launch configuration the bench times: a plan made with GA_PLAN_KV_E4M3,
    whose units the planner makes 4 kv heads wide."""
    wl = W.config(5)
    fam = wl.local
    assert fam.kv_dtype == W.KV_E4M3
    fi = W.make_family_inputs(wl, fam, device=DEV, poison=True, release_old=True)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=256, window=fam.window,
                             flags=ga.GA_PLAN_KV_E4M3)
    assert plan.kv_heads_per_unit == 4                    # the planner's own choice here
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 16)
    assert_close(out[rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                 kv_dtype=1, what="ragged local E4M3 4-head units")
    del fi
    torch.cuda.empty_cache()
