"""Randomised parity: many seeded shapes against the oracle (E4M3 pools
twice: with a plain plan and with one made for E4M3 pools), plus the
call-level options (external combine, side streams, no error word)."""
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"
EDGE_LENS = [0, 1, 15, 16, 17, 31, 32, 33, 1023, 1024, 1025, 2047, 2048, 2049]


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _case(seed):
    rng = np.random.default_rng(seed)
    D = int(rng.choice([256, 512]))
    kv = int(rng.choice([0, 1]))
    Hkv = int(rng.choice([1, 2, 3, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16, 24]))
    # hd256 goes through the windowed entry (a window beyond every length is
    # full context); hd512 through the global one
    window = int(rng.choice([1, 7, 64, 200, 1024, 1 << 20])) if D == 256 else 0
    B = int(rng.integers(1, 24))
    lens = rng.integers(0, 2600, size=B)
    pick = rng.random(B) < 0.4
    lens[pick] = rng.choice(EDGE_LENS, size=int(pick.sum()))
    split = [dict(requested_splits=1), dict(requested_splits=int(rng.integers(2, 9))),
             dict(fixed_chunk_tokens=16 * int(rng.integers(1, 20))), dict()][int(rng.integers(0, 4))]
    scale = float(rng.choice([1.0 / math.sqrt(D), 0.5 / math.sqrt(D), 0.02]))
    fam = W.Family("local" if window else "global", g * Hkv, Hkv, D, window, kv)
    return fam, lens.astype(np.int32), split, scale


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes(ga, seed):
    fam, lens, split, scale = _case(seed)
    wl = W.Workload("fuzz", lens, 16, fam, fam)
    fi = W.make_family_inputs(wl, fam, device=DEV, seed=seed, poison=True,
                              release_old=bool(fam.window) and seed % 2 == 0)
    ref = oracle_decode(fi, scale=scale)
    # E4M3 pools: a plain plan and one made for them (16-column units above 8
    # query heads per kv head, several kv heads per sliding unit when they fill)
    for flags in ((0, ga.GA_PLAN_KV_E4M3) if fam.kv_dtype else (0,)):
        plan = ga.ga_plan_splits(lens, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, flags=flags, **split)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = run_decode(ga, fi, plan, scale=scale, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        what = f"seed {seed}: D={fam.head_dim} kv={fam.kv_dtype} " \
               f"g={fam.num_q_heads // fam.num_kv_heads} Hkv={fam.num_kv_heads} " \
               f"W={fam.window} B={len(lens)} {split} flags={flags} col_tile={plan.col_tile}"
        got = out.float().cpu().numpy()
        assert_close(got, ref, kv_dtype=fam.kv_dtype, what=what)
    assert np.all(got[lens == 0] == 0)


def test_external_combine_is_bit_identical(ga):
    wl = W.config(2)
    fi = W.make_family_inputs(wl, wl.global_, device=DEV, poison=True)
    kw = dict(num_q_heads=16, num_kv_heads=2, head_dim=512, window=0, fixed_chunk_tokens=256)
    inner = ga.ga_plan_splits(wl.seq_lens, **kw)
    outer = ga.ga_plan_splits(wl.seq_lens, flags=ga.GA_PLAN_EXTERNAL_COMBINE, **kw)
    a = run_decode(ga, fi, inner).clone()
    ws = ga.workspace_for(outer, DEV)
    b = torch.full_like(fi.q, float("nan"))
    run_decode(ga, fi, outer, workspace=ws, out=b)
    po, plse, _ = ga.workspace_views(outer, ws)
    ga.ga_splitkv_combine(po, plse, outer, fi.seq_lens, fi.page_table.shape[1], b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_side_stream_and_no_error_word(ga):
    wl = W.config(1)
    results = []
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, device=DEV, poison=True)
        plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, requested_splits=2)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            out = run_decode(ga, fi, plan, err=None)
        s.synchronize()
        results.append((out.float().cpu().numpy(), oracle_decode(fi)))
    for got, ref in results:
        assert_close(got, ref, what="side stream")
