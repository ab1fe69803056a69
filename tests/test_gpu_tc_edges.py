"""GPU parity at the edges of the tensor-core E4M3 sliding-window decode.

That kernel streams a unit's pages in groups of 8 ("superstages", 128 keys:
one MMA tile) and multiplies V in steps of two pages, so its own edge cases
are page counts around multiples of 8 and odd counts (the page after an odd
last one is read by the PV step and must hold zeros), head groups narrower
than the compiled column count, split chunks that cut superstages, a page id
flagged invalid in the middle of a superstage, and NaN in slots no query
attends.  The method is the paged sliding-window attention over an E4M3 pool
("[Model] Gemma 4 M2 26B-A4B", Proposed Plan: opt-in FP8 pool for the sliding
family; "[Model] Gemma 4 M3 31B", Acceptance Criteria: window boundaries);
outputs are compared with the fp64 oracle run on the same stored codes.
"""
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = 16

# page counts 1, 7, 8, 9, 15, 16, 17, 64, 65 with keys ending mid-page and on a page edge
EDGE_LENS = [1, 16, 7 * P - 3, 8 * P, 8 * P + 1, 9 * P - 5, 15 * P, 16 * P, 16 * P + 9,
             17 * P - 1, 64 * P, 1023, 1024, 1025, 65 * P - 2]


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _inputs(lens, Hq, Hkv, window, seed):
    fam = W.Family("local", Hq, Hkv, 256, window, 1)
    wl = W.Workload("tc-edges", np.asarray(lens, dtype=np.int32), P, fam, fam)
    return W.make_family_inputs(wl, fam, device=DEV, seed=seed, poison=True)


def _plan(ga, fi, **kw):
    fam = fi.family
    return ga.ga_plan_splits(fi.seq_lens.cpu().numpy(), num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=256, window=fam.window, **kw)


@pytest.mark.parametrize("window", [1 << 20, 1024, 40])
@pytest.mark.parametrize("g", [1, 2, 3, 5, 8, 12, "12-e4m3-plan"])
def test_superstage_edges(ga, window, g):
    """Every page count around a superstage, every column-count variant
    (1..2 -> 2 columns, 3..4 -> 4, more -> 8; 12 -> two head groups, or one
    16-column unit with a plan made with GA_PLAN_KV_E4M3), three split modes;
    unattended slots hold NaN."""
    flags = ga.GA_PLAN_KV_E4M3 if g == "12-e4m3-plan" else 0
    g = 12 if flags else g
    Hkv = 2
    fi = _inputs(EDGE_LENS, g * Hkv, Hkv, window, seed=300 + g)
    ref = oracle_decode(fi)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for split in (dict(requested_splits=1), dict(fixed_chunk_tokens=3 * P),
                  dict(requested_splits=3)):
        plan = _plan(ga, fi, flags=flags, **split)
        assert (plan.col_tile == 16) == bool(flags)
        out = run_decode(ga, fi, plan, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.float().cpu().numpy(), ref, kv_dtype=1,
                     what=f"window {window} g {g} {split}")


def test_flagged_page_mid_superstage(ga):
    """A page id outside the pool in the middle of a superstage is reported
    and not read; the other rows are exact and nothing turns NaN."""
    fi = _inputs([20 * P, 300, 13 * P + 4], 4, 2, 1 << 20, seed=321)
    fi.page_table[0, 11] = 1 << 30                       # logical page 11: superstage 1, slot 3
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_decode(ga, fi, _plan(ga, fi), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_PAGE_ID
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert_close(got[1:], oracle_decode(fi, rows=[1, 2]), kv_dtype=1, what="unflagged rows")


def test_scale_one_peaked_softmax(ga):
    """Scale 1.0 (the Gemma convention) makes the softmax peaked, so the
    running max is raised and O rescaled in tensor memory many times."""
    fi = _inputs(EDGE_LENS, 4, 2, 1024, seed=333)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_decode(ga, fi, _plan(ga, fi), err=err, scale=1.0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle_decode(fi, scale=1.0)
    # bf16 output: half an ulp of the largest |o| on top of the E4M3 bound
    extra = 0.5 * 2.0 ** (math.floor(math.log2(max(np.abs(ref).max(), 1e-30))) - 7)
    assert_close(out.float().cpu().numpy(), ref, kv_dtype=1, what="scale 1.0", extra_abs=extra)
