"""Multi-query decode (S query tokens per row, causal inside the chunk) through
the C ABI against the oracle: small cases over edge lengths, every split mode
and both KV types; column layouts that span several head groups; chunk parity
against one-query decodes on the GPU; the 31B-shaped batch at S = 4 (an
EAGLE3 verify step: 3 speculative tokens + 1, "Gemma 4 31B on vLLM", LIGHT
recipe)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close

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


def _inputs(lens, fam, S, seed, poison=True, wl=None):
    """Pools for a row set whose S queries attend the union of their windows
    (W + S - 1 keys for the sliding family): pages are kept / poisoned by that
    union, q is [B, Hq, S, D]."""
    alloc = dataclasses.replace(fam, window=fam.window + S - 1 if fam.window else 0)
    if wl is None:
        wl = W.Workload("mq", np.asarray(lens, dtype=np.int32), 16, alloc, alloc)
    fi = W.make_family_inputs(wl, alloc, device=DEV, seed=seed, poison=poison,
                              release_old=fam.window > 0)
    g = torch.Generator().manual_seed(seed + 1000)
    q = torch.randn(len(lens), fam.num_q_heads, S, fam.head_dim, generator=g).to(torch.bfloat16)
    return fi, q.to(DEV)


def _plan(ga, lens, fam, S, **kw):
    return ga.ga_plan_splits_mq(lens, q_len=S, num_q_heads=fam.num_q_heads,
                                num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                window=fam.window, **kw)


def _decode(ga, fi, q, fam, plan, err=None, scale=None):
    scale = 1.0 / math.sqrt(fam.head_dim) if scale is None else scale
    out = torch.full_like(q, float("nan"))
    kw = dict(scale=scale, plan=plan, workspace=ga.workspace_for(plan, DEV), out=out,
              k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    if fam.window:
        return ga.ga_decode_local_hd256(q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                        window=fam.window, **kw)
    return ga.ga_decode_global_hd512(q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)


def _oracle(fi, q, fam, scale=None, rows=None):
    scale = 1.0 / math.sqrt(fam.head_dim) if scale is None else scale
    ks = None if fi.k_scale is None else fi.k_scale.cpu()
    vs = None if fi.v_scale is None else fi.v_scale.cpu()
    if rows is None:
        return O.decode_mq(q.cpu(), fi.k_pool.cpu(), fi.v_pool.cpu(), fi.page_table.cpu(),
                           fi.seq_lens.cpu(), num_kv_heads=fam.num_kv_heads, window=fam.window,
                           scale=scale, kv_dtype=fam.kv_dtype, k_scale=ks, v_scale=vs)
    # only the pages the sampled rows reference, renumbered
    table = fi.page_table[rows].cpu().numpy()
    used = np.unique(table[table >= 0])
    remap = np.full(max(int(fi.num_pages), 1), -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    sub = np.where(table >= 0, remap[np.maximum(table, 0)], -1).astype(np.int32)
    idx = torch.as_tensor(used, device=fi.k_pool.device)
    return O.decode_mq(q[rows].cpu(), fi.k_pool.index_select(0, idx).cpu(),
                       fi.v_pool.index_select(0, idx).cpu(), torch.from_numpy(sub),
                       fi.seq_lens[rows].cpu(), num_kv_heads=fam.num_kv_heads,
                       window=fam.window, scale=scale, kv_dtype=fam.kv_dtype, k_scale=ks,
                       v_scale=vs, nthreads=8)


EDGE = [0, 1, 3, 4, 5, 16, 17, 31, 33, 47, 120, 300]
FAMS = {"local": W.Family("local", 8, 4, 256, 32), "global": W.Family("global", 16, 2, 512, 0)}
SPLITS = {"none": dict(requested_splits=1), "count3": dict(requested_splits=3),
          "chunk32": dict(fixed_chunk_tokens=32), "auto": dict()}


@pytest.mark.parametrize("split", sorted(SPLITS))
@pytest.mark.parametrize("kv", [0, 1])
@pytest.mark.parametrize("family", ["local", "global"])
@pytest.mark.parametrize("S", [2, 4])
def test_mq_parity_edge_lengths(ga, err, S, family, kv, split):
    fam = dataclasses.replace(FAMS[family], kv_dtype=kv)
    fi, q = _inputs(EDGE, fam, S, seed=S * 10 + kv)
    plan = _plan(ga, EDGE, fam, S, **SPLITS[split])
    out = _decode(ga, fi, q, fam, plan, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.float().cpu().numpy()
    assert_close(got, _oracle(fi, q, fam), kv_dtype=kv, what=f"S={S} {family} kv={kv} {split}")
    # queries at negative positions (rows shorter than S) give zeros
    for b, L in enumerate(EDGE):
        for i in range(S):
            if L - S + i < 0:
                assert np.all(got[b, :, i] == 0)


@pytest.mark.parametrize("Hq,Hkv,D,window,S", [
    (3, 3, 256, 40, 3),        # g = 1: 3 columns per kv head
    (6, 2, 256, 24, 3),        # g = 3, S = 3: 9 columns -> 2 head groups
    (8, 4, 256, 64, 8),        # g = 2, S = 8: 16 columns -> 2 groups
    (16, 2, 512, 0, 3),        # g = 8, S = 3: 24 columns -> 3 groups
    (8, 1, 512, 0, 16),        # g = 8, S = 16: 128 columns -> 16 groups
])
def test_mq_column_groups(ga, err, Hq, Hkv, D, window, S):
    fam = W.Family("local" if window else "global", Hq, Hkv, D, window)
    lens = [2, 19, 77, 160, 33]
    fi, q = _inputs(lens, fam, S, seed=7 + S)
    plan = _plan(ga, lens, fam, S, requested_splits=2)
    out = _decode(ga, fi, q, fam, plan, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.float().cpu().numpy(), _oracle(fi, q, fam),
                 what=f"Hq={Hq} Hkv={Hkv} D={D} W={window} S={S}")


@pytest.mark.parametrize("family", ["local", "global"])
def test_mq_chunk_parity_with_one_query_decodes(ga, err, family):
    """Query i of an S-token chunk matches a one-query decode of the same row
    cut at length L - S + i + 1 ("visible-cx/Gemma-4-31B-CoreAI",
    hybrid-pf64/ bundles: chunked and token-by-token walks must agree)."""
    fam = FAMS[family]
    S = 4
    lens = [40, 200, 1030, 5, 64]
    fi, q = _inputs(lens, fam, S, seed=21, poison=False)
    out = _decode(ga, fi, q, fam, _plan(ga, lens, fam, S), err).float().cpu()
    for i in range(S):
        cut = torch.clamp(fi.seq_lens - S + i + 1, min=0).to(torch.int32)
        one_plan = ga.ga_plan_splits(cut.cpu().numpy(), num_q_heads=fam.num_q_heads,
                                     num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                     window=fam.window)
        fi1 = dataclasses.replace(fi, seq_lens=cut.to(DEV).contiguous())
        q1 = q[:, :, i].contiguous()
        one = _decode(ga, fi1, q1, fam, one_plan, err).float().cpu()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # both sides are rounded to bf16 on their own: a value near a rounding
        # boundary may land one ulp (of the largest |o|) apart
        ref = one.numpy().astype(np.float64)
        ulp = 2.0 ** (math.floor(math.log2(max(np.abs(ref).max(), 1e-30))) - 7)
        assert_close(out[:, :, i].numpy(), ref, what=f"{family} query {i} vs one-query decode",
                     extra_abs=ulp)


@pytest.mark.parametrize("kv", [0, 1], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("family", ["local", "global"])
def test_mq_31b_eagle_verify_sampled(ga, err, family, kv):
    """31B-shaped batch, S = 4 (3 speculative tokens + the accepted one), the
    planner's plan, sampled rows against the oracle; also on E4M3 pools with
    a plan made for them ("Gemma 4 31B on vLLM -- operating-point reference",
    LIGHT recipe: an fp8 KV cache with EAGLE3 verify)."""
    wl = W.config(3)
    fam = wl.local if family == "local" else wl.global_
    fam = dataclasses.replace(fam, kv_dtype=kv)
    S = 4
    alloc = dataclasses.replace(fam, window=fam.window + S - 1 if fam.window else 0)
    wl2 = W.Workload(wl.name, wl.seq_lens, wl.page_size, alloc, alloc)
    fi, q = _inputs(wl.seq_lens, fam, S, seed=0, poison=False, wl=wl2)
    flags = ga.GA_PLAN_KV_E4M3 if kv else 0
    out = _decode(ga, fi, q, fam, _plan(ga, wl.seq_lens, fam, S, flags=flags), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 4)
    ref = _oracle(fi, q, fam, rows=rows)
    assert_close(out[rows].float().cpu().numpy(), ref, kv_dtype=kv, what=f"31B S=4 {family}")
    del fi
    torch.cuda.empty_cache()


def test_mq_shape_must_match_plan(ga):
    fam = FAMS["local"]
    lens = [40, 33]
    fi, q = _inputs(lens, fam, 4, seed=3)
    plan = _plan(ga, lens, fam, 2)            # plan for S = 2, q has S = 4
    with pytest.raises(ga.GAError):
        _decode(ga, fi, q, fam, plan)
