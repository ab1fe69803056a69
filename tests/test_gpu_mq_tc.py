"""GPU parity of the tensor-core multi-query decode against the fp64 oracle.

Plans with units of 64 (query, head) columns (the default from 32 columns
per kv head at hd512 and 64 at hd256, or any count above 8 with
GA_PLAN_TENSOR_CORE_UNITS) run on bf16 pools in a kernel whose products run
on tcgen05, 128 keys (8 pages) per stage.  That kernel's own edge cases are:
- lengths around 128-key stages and 16-key pages;
- rows shorter than S (queries at negative positions);
- column tiles that are partly empty (g * S not a multiple of 64);
- several tiles per kv head;
- the causal edge inside the last stage;
- the sliding window's edge for every query of the chunk;
- split chunks that cut stages;
- a page id flagged invalid in the middle of a stage;
- NaN in slots no query attends;
- a peaked softmax (scale 1.0) that raises the running maxima, and so
  rescales O in tensor memory, many times.

The method is the paged attention of both families with the S queries of a
row as extra columns, each with its causal and window mask
("visible-cx/Gemma-4-31B-CoreAI" model card, hybrid-pf64/ bundles: prefill
chunks of 64 tokens; "Gemma 4 31B on vLLM -- operating-point reference",
Operating-point recipes, LIGHT: speculative verify).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close
from tests.test_gpu_mq import _decode, _inputs, _oracle, _plan

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = 16

# pages / stages: 1 key, mid first page, one stage - 1 / exact / + 1, two
# stages around their edge, a long row with a ragged last page
EDGE_TC = [1, 5, 63, 64, 65, 127, 128, 129, 250, 256, 257, 700]
FAMS = {"local": W.Family("local", 8, 4, 256, 96),     # g = 2
        "global": W.Family("global", 16, 2, 512, 0)}   # g = 8
SPLITS = {"none": dict(requested_splits=1), "count3": dict(requested_splits=3),
          "chunk64": dict(fixed_chunk_tokens=64), "auto": dict()}


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


@pytest.fixture()
def err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _tc_plan(ga, lens, fam, S, **kw):
    """A plan with 64-column tensor-core units whatever the column count."""
    return _plan(ga, lens, fam, S, flags=ga.GA_PLAN_TENSOR_CORE_UNITS, **kw)


def _check(ga, err, fi, q, fam, plan, ref, what, scale=None, extra_abs=None):
    assert plan.col_tile == 64, "plan does not use the tensor-core units"
    out = _decode(ga, fi, q, fam, plan, err, scale=scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error word {int(err.item())}"
    got = out.float().cpu().numpy()
    assert_close(got, ref, what=what, extra_abs=extra_abs)
    return got


@pytest.mark.parametrize("family", ["local", "global"])
@pytest.mark.parametrize("S", [8, 16, 64])
def test_tc_edge_lengths_every_split(ga, err, S, family):
    """Every edge length, four split modes, one oracle run; queries at
    negative positions give zeros."""
    fam = FAMS[family]
    fi, q = _inputs(EDGE_TC, fam, S, seed=400 + S)
    ref = _oracle(fi, q, fam)
    for name, split in SPLITS.items():
        got = _check(ga, err, fi, q, fam, _tc_plan(ga, EDGE_TC, fam, S, **split), ref,
                     f"S={S} {family} {name}")
        for b, L in enumerate(EDGE_TC):
            for i in range(S):
                if L - S + i < 0:
                    assert np.all(got[b, :, i] == 0)


@pytest.mark.parametrize("Hq,Hkv,D,window,S", [
    (6, 2, 256, 40, 7),        # g = 3: 21 columns, one tile, 43 columns empty
    (16, 2, 512, 0, 9),        # g = 8: 72 columns -> tiles of 64 and 8
    (4, 1, 512, 0, 40),        # g = 4: 160 columns -> 64, 64, 32
    (2, 1, 256, 1000, 33),     # g = 2: 66 columns -> 64 and 2; window longer than rows
    (32, 4, 512, 0, 2),        # g = 8, S = 2: 16 columns (the smallest tensor-core case)
])
def test_tc_partial_and_multiple_tiles(ga, err, Hq, Hkv, D, window, S):
    fam = W.Family("local" if window else "global", Hq, Hkv, D, window)
    lens = [3, 40, 129, 300, 77, 1]
    fi, q = _inputs(lens, fam, S, seed=11 + S)
    ref = _oracle(fi, q, fam)
    for split in (dict(requested_splits=1), dict(requested_splits=2)):
        _check(ga, err, fi, q, fam, _tc_plan(ga, lens, fam, S, **split), ref,
               f"Hq={Hq} Hkv={Hkv} D={D} W={window} S={S} {split}")


@pytest.mark.parametrize("family", ["local", "global"])
def test_tc_flagged_page_mid_stage(ga, err, family):
    """A page id outside the pool in the middle of a stage is reported and
    not read; the other rows are exact and nothing turns NaN."""
    fam = FAMS[family]
    S = 16
    lens = [20 * P, 300, 13 * P + 4]
    fi, q = _inputs(lens, fam, S, seed=77)
    # a page the row's union window still attends, slot 3 of a stage
    first = int(fi.seq_lens[0].item() - 1) // P
    bad = first - 4
    fi.page_table[0, bad] = 1 << 30
    out = _decode(ga, fi, q, fam, _tc_plan(ga, lens, fam, S, requested_splits=1), err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_PAGE_ID
    got = out.float().cpu().numpy()
    assert np.isfinite(got).all()
    ref = _oracle(fi, q, fam, rows=[1, 2])
    assert_close(got[1:], ref, what=f"{family} unflagged rows")


@pytest.mark.parametrize("family", ["local", "global"])
def test_tc_scale_one_peaked_softmax(ga, err, family):
    """Scale 1.0 (the Gemma convention) makes the softmax peaked: the running
    maxima rise past the slack often and O is rescaled in tensor memory."""
    fam = FAMS[family]
    S = 16
    fi, q = _inputs(EDGE_TC, fam, S, seed=91)
    ref = _oracle(fi, q, fam, scale=1.0)
    # bf16 output: half an ulp of the largest |o| on top of the bf16 bound
    extra = 0.5 * 2.0 ** (math.floor(math.log2(max(np.abs(ref).max(), 1e-30))) - 7)
    _check(ga, err, fi, q, fam, _tc_plan(ga, EDGE_TC, fam, S), ref, f"{family} scale 1.0",
           scale=1.0, extra_abs=extra)


@pytest.mark.parametrize("family", ["local", "global"])
def test_tc_31b_prefill_chunk_sampled(ga, err, family):
    """31B-shaped batch with a 64-token prefill chunk per row (S = 64: 512
    columns per global kv head, 128 per local one), the planner's plan,
    sampled rows against the oracle."""
    wl = W.config(3)
    fam = wl.local if family == "local" else wl.global_
    S = 64
    alloc = dataclasses.replace(fam, window=fam.window + S - 1 if fam.window else 0)
    wl2 = W.Workload(wl.name, wl.seq_lens, wl.page_size, alloc, alloc)
    fi, q = _inputs(wl.seq_lens, fam, S, seed=0, poison=False, wl=wl2)
    plan = _plan(ga, wl.seq_lens, fam, S)
    assert plan.col_tile == 64
    out = _decode(ga, fi, q, fam, plan, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 2)
    ref = _oracle(fi, q, fam, rows=rows)
    assert_close(out[rows].float().cpu().numpy(), ref, what=f"31B S=64 {family}")
    del fi
    torch.cuda.empty_cache()
