"""E4M3 pools with more than 8 (query, head) columns per kv head: a plan made
with GA_PLAN_KV_E4M3 asks the tcgen05 E4M3 decode for units of 16 columns
(col_tile 16: S queries x g query heads of a kv head, its pages streamed once
for 16 columns instead of once per 8).  Checked against the oracle over edge
lengths, every split mode, both head dims, K == V pools, more than one
16-column unit per kv head, a ragged last unit, a GQA group of 16 at one
query per row, a page id flagged invalid mid-superstage, scale 1.0 (a peaked
softmax), and a 31B-shaped batch at S = 2 ("Gemma 4 31B on vLLM --
operating-point reference", LIGHT recipe: an fp8 KV cache under EAGLE3
verify; "[Model] Gemma 4 M3 31B", Acceptance Criteria: windows of 1024)."""
import dataclasses

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close
from tests.test_gpu_mq import EDGE, SPLITS, _decode, _inputs, _oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


@pytest.fixture()
def err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# (family, S): columns per kv head = g x S
SHAPES = {
    "global_g8_S2": (W.Family("global", 16, 2, 512, 0, 1), 2),     # 16: one unit
    "global_g8_S3": (W.Family("global", 16, 2, 512, 0, 1), 3),     # 24: 16 + 8 valid
    "global_g8_S4": (W.Family("global", 16, 2, 512, 0, 1), 4),     # 32: two units
    "global_g16_S1": (W.Family("global", 32, 2, 512, 0, 1), 1),    # 16 query heads, one query
    "local_g8_S2": (W.Family("local", 16, 2, 256, 32, 1), 2),      # 16
    "local_g2_S8": (W.Family("local", 8, 4, 256, 32, 1), 8),       # 16
    "local_g4_S3": (W.Family("local", 8, 2, 256, 1024, 1), 3),     # 12: one unit, 4 idle columns
}


def _plan(ga, lens, fam, S, **kw):
    return ga.ga_plan_splits_mq(lens, q_len=S, num_q_heads=fam.num_q_heads,
                                num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                window=fam.window, flags=ga.GA_PLAN_KV_E4M3, **kw)


def _check(ga, err, fam, S, lens, fi, q, plan, what):
    out = _decode(ga, fi, q, fam, plan, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, what
    got = out.float().cpu().numpy()
    assert_close(got, _oracle(fi, q, fam), kv_dtype=fam.kv_dtype, what=what)
    for b, L in enumerate(lens):              # queries before position 0 give zeros
        for i in range(S):
            if L - S + i < 0:
                assert np.all(got[b, :, i] == 0), what
    return got


@pytest.mark.parametrize("split", sorted(SPLITS))
@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_wide_units_edge_lengths(ga, err, shape, split):
    fam, S = SHAPES[shape]
    plan = _plan(ga, EDGE, fam, S, **SPLITS[split])
    cols = fam.num_q_heads // fam.num_kv_heads * S
    assert plan.col_tile == 16 and plan.kv_heads_per_unit == 1
    assert plan.units == plan.row_chunks * fam.num_kv_heads * -(-cols // 16)
    fi, q = _inputs(EDGE, fam, S, seed=101 + S)
    _check(ga, err, fam, S, EDGE, fi, q, plan, f"{shape} {split}")


@pytest.mark.parametrize("shape", ["global_g8_S4", "local_g2_S8"])
def test_wide_units_kv_alias(ga, err, shape):
    """One pool for K and V (same pointer): every block fetched once into a V
    slot that serves both products."""
    fam, S = SHAPES[shape]
    lens = [0, 5, 17, 64, 333, 1100]
    fi, q = _inputs(lens, fam, S, seed=7)
    fi = dataclasses.replace(fi, v_pool=fi.k_pool, v_scale=fi.k_scale)
    for split in (dict(requested_splits=1), dict(requested_splits=3)):
        plan = _plan(ga, lens, fam, S, **split)
        assert plan.col_tile == 16
        _check(ga, err, fam, S, lens, fi, q, plan, f"{shape} alias {split}")


def test_wide_units_against_eight_column_units(ga, err):
    """The same inputs through 16-column units and through 8-column ones (a
    plan made without GA_PLAN_KV_E4M3): both within tolerance of the
    oracle."""
    fam, S = SHAPES["global_g8_S4"]
    lens = [1, 16, 48, 700, 2049]
    fi, q = _inputs(lens, fam, S, seed=3)
    wide = _plan(ga, lens, fam, S, requested_splits=2)
    narrow = ga.ga_plan_splits_mq(lens, q_len=S, num_q_heads=fam.num_q_heads,
                                  num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                  window=0, requested_splits=2)
    assert wide.col_tile == 16 and narrow.col_tile != 16
    a = _check(ga, err, fam, S, lens, fi, q, wide, "16-column units")
    b = _check(ga, err, fam, S, lens, fi, q, narrow, "8-column units")
    assert_close(a, b.astype(np.float64), kv_dtype=fam.kv_dtype, what="16 vs 8 columns")


def test_wide_units_31b_s2_sampled(ga, err):
    """31B-shaped global family on E4M3 pools at S = 2 (one 16-column unit per
    kv head) with the planner's plan, sampled rows against the oracle."""
    wl = W.config(3)
    fam = dataclasses.replace(wl.global_, kv_dtype=W.KV_E4M3)
    S = 2
    fi, q = _inputs(wl.seq_lens, fam, S, seed=0, poison=False)
    plan = _plan(ga, wl.seq_lens, fam, S)
    assert plan.col_tile == 16
    out = _decode(ga, fi, q, fam, plan, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 4)
    assert_close(out[rows].float().cpu().numpy(), _oracle(fi, q, fam, rows=rows),
                 kv_dtype=fam.kv_dtype, what="31B global S=2 E4M3")
    del fi
    torch.cuda.empty_cache()


def test_wide_units_flagged_page(ga):
    """A page id outside the pool in the middle of a superstage, in a
    16-column unit at head_dim 512 (both half-warps at work): reported, not
    read; the other rows within tolerance and nothing turns NaN."""
    from tests.helpers import oracle_decode, run_decode
    fam = W.Family("global", 32, 2, 512, 0, W.KV_E4M3)          # group 16, one query
    lens = [20 * 16, 300, 13 * 16 + 4]
    wl = W.Workload("wide-flag", np.asarray(lens, dtype=np.int32), 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=77, poison=True)
    fi.page_table[0, 6] = 1 << 30                 # logical page 6: superstage 1, page 2
    plan = ga.ga_plan_splits(lens, num_q_heads=32, num_kv_heads=2, head_dim=512, window=0,
                             flags=ga.GA_PLAN_KV_E4M3)
    assert plan.col_tile == 16
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_PAGE_ID
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got[1:], oracle_decode(fi, rows=[1, 2]), kv_dtype=fam.kv_dtype,
                 what="unflagged rows")


@pytest.mark.parametrize("shape", ["global_g8_S2", "local_g2_S8"])
def test_wide_units_scale_one(ga, err, shape):
    """Scale 1.0 (the Gemma convention): a peaked softmax whose running maxima
    are raised, and O^T rescaled in tensor memory, many times per unit."""
    import math
    fam, S = SHAPES[shape]
    lens = [3, 40, 333, 1030, 2049]
    fi, q = _inputs(lens, fam, S, seed=55)
    plan = _plan(ga, lens, fam, S, requested_splits=2)
    assert plan.col_tile == 16
    out = _decode(ga, fi, q, fam, plan, err, scale=1.0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _oracle(fi, q, fam, scale=1.0)
    extra = 0.5 * 2.0 ** (math.floor(math.log2(max(np.abs(ref).max(), 1e-30))) - 7)
    assert_close(out.float().cpu().numpy(), ref, kv_dtype=fam.kv_dtype,
                 what=f"{shape} scale 1.0", extra_abs=extra)
