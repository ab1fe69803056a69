"""The split-KV merge behind every decode kernel (page-parallel bf16, E4M3 on
tcgen05 at both head dims, K == V, column-parallel units, the tcgen05
multi-query kernel): the decode call's own merge must give the same bits as a
decode with an external combine followed by ga_splitkv_combine, repeat calls
must give the same bits, and both must match the oracle.  Rows with more than
64 chunks take the merge's per-thread form; a workspace may serve plans of
different shapes in turn.  ("visible-cx/Gemma-4-31B-CoreAI", "--metal-sdpa is
mandatory here": flash-decode split and merge.)"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    "local_bf16": (W.Family("local", 16, 8, 256, 1024), 1),
    "global_bf16": (W.Family("global", 16, 2, 512, 0), 1),
    "local_e4m3": (W.Family("local", 16, 8, 256, 1024, 1), 1),     # tcgen05, hd256
    "global_e4m3": (W.Family("global", 16, 2, 512, 0, 1), 1),      # tcgen05, hd512
    "global_bf16_kv_alias": (W.Family("global", 16, 2, 512, 0), 1),
    "local_bf16_5_queries": (W.Family("local", 16, 8, 256, 1024), 5),   # column-parallel
    "global_bf16_8_queries": (W.Family("global", 16, 2, 512, 0), 8),    # tcgen05 multi-query
}


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _setup(case, seed=11):
    fam, S = CASES[case]
    lens = np.array([1500, 3000, 40, 1025, 16, 0, 2222, 700], dtype=np.int32)
    alloc = dataclasses.replace(fam, window=fam.window + S - 1 if fam.window else 0)
    wl = W.Workload("merge", lens, 16, alloc, alloc)
    fi = W.make_family_inputs(wl, alloc, device=DEV, seed=seed, poison=True,
                              release_old=fam.window > 0)
    if case.endswith("kv_alias"):
        fi = dataclasses.replace(fi, v_pool=fi.k_pool, v_scale=fi.k_scale)
    if S > 1:
        g = torch.Generator().manual_seed(seed + 3)
        q = torch.randn(len(lens), fam.num_q_heads, S, fam.head_dim, generator=g)
        fi = dataclasses.replace(fi, q=q.to(torch.bfloat16).to(DEV))
    return fam, S, lens, dataclasses.replace(fi, family=fam)


def _call(ga, fi, plan, ws, out, err):
    fam = fi.family
    kw = dict(scale=1.0 / math.sqrt(fam.head_dim), plan=plan, workspace=ws, out=out,
              k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    if fam.window:
        ga.ga_decode_local_hd256(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                 window=fam.window, **kw)
    else:
        ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                  **kw)
    return out


@pytest.mark.parametrize("split", [dict(requested_splits=3), dict(fixed_chunk_tokens=64)],
                         ids=["s3", "c64"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_internal_equals_external_combine(ga, case, split):
    fam, S, lens, fi = _setup(case)
    kw = dict(num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
              head_dim=fam.head_dim, window=fam.window, q_len=S, **split)
    inner = ga.ga_plan_splits(lens, **kw)
    outer = ga.ga_plan_splits(lens, flags=ga.GA_PLAN_EXTERNAL_COMBINE, **kw)
    assert inner.mode != ga.GA_SPLIT_NONE
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = ga.workspace_for(inner, DEV)
    a = _call(ga, fi, inner, ws, torch.full_like(fi.q, float("nan")), err)
    a2 = _call(ga, fi, inner, ws, torch.full_like(fi.q, float("nan")), err)
    ws2 = ga.workspace_for(outer, DEV)
    b = _call(ga, fi, outer, ws2, torch.full_like(fi.q, float("nan")), err)
    po, plse, _ = ga.workspace_views(outer, ws2)
    ga.ga_splitkv_combine(po, plse, outer, fi.seq_lens, fi.page_table.shape[1], b, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(a, a2)
    assert torch.equal(a, b), f"{case}: the call's merge differs from the external one"
    scale = 1.0 / math.sqrt(fam.head_dim)
    if S == 1:
        ref = oracle_decode(fi)
    else:
        ref = O.decode_mq(fi.q.cpu(), fi.k_pool.cpu(), fi.v_pool.cpu(), fi.page_table.cpu(),
                          fi.seq_lens.cpu(), num_kv_heads=fam.num_kv_heads, window=fam.window,
                          scale=scale, kv_dtype=fam.kv_dtype,
                          k_scale=None if fi.k_scale is None else fi.k_scale.cpu(),
                          v_scale=None if fi.v_scale is None else fi.v_scale.cpu())
    assert_close(a.float().cpu().numpy(), ref, kv_dtype=fam.kv_dtype, what=case)


@pytest.mark.parametrize("case", ["local_bf16", "global_bf16"])
def test_more_than_64_chunks_per_row(ga, case):
    """16-token chunks: rows with more than 64 attended pages (up to 188 here)
    have more chunks than the warp merge's 64 and take the per-thread merge."""
    fam, S, lens, fi = _setup(case)
    plan = ga.ga_plan_splits(lens, num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
                             head_dim=fam.head_dim, window=fam.window, fixed_chunk_tokens=16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _call(ga, fi, plan, ga.workspace_for(plan, DEV), torch.full_like(fi.q, float("nan")),
                err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    def pages(L):              # logical pages holding the attended keys of a row
        lo = max(0, L - fam.window) if fam.window else 0
        return (L - 1) // 16 - lo // 16 + 1 if L > 0 else 0
    assert max(pages(int(L)) for L in lens) > 64
    assert_close(out.float().cpu().numpy(), oracle_decode(fi), what=case)


def test_workspace_shared_by_plans_of_different_shapes(ga):
    """One workspace serves a local and a global plan in turn (different
    batch sizes and head counts); every call matches the oracle."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cases = []
    for case, lens in (("local_bf16", [1500, 3000, 40, 1025]),
                       ("global_bf16", [1500, 3000, 40, 1025, 16, 0, 2222, 700])):
        fam, S, _, _ = _setup(case)
        lens = np.asarray(lens, dtype=np.int32)
        wl = W.Workload("share", lens, 16, fam, fam)
        fi = W.make_family_inputs(wl, fam, device=DEV, seed=21, poison=True,
                                  release_old=fam.window > 0)
        plan = ga.ga_plan_splits(lens, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, requested_splits=4)
        cases.append((fi, plan))
    ws = torch.empty(max(p.workspace_bytes for _, p in cases), dtype=torch.uint8, device=DEV)
    for rnd in range(2):
        for fi, plan in cases:
            out = _call(ga, fi, plan, ws, torch.full_like(fi.q, float("nan")), err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert_close(out.float().cpu().numpy(), oracle_decode(fi),
                         what=f"{fi.family.name} round {rnd}")
