"""The decode entry point that allocates nothing.

ga_decode_global_hd512_noalloc serves callers that cannot allocate device
memory at decode time (for example a plain-C serving loop without a caching
allocator, where cudaMalloc would synchronise the device mid-step, or a host
whose free device memory all went to fixed KV pools).  Its split-KV scratch is
a device array built into the library.  These tests call it through the C ABI
and check it, on two calls in a row, against ga_decode_global_hd512 given its
own workspace (the same kernel on the same plan: the outputs must be
identical) and against the fp64 oracle; plans that need more scratch than the
array holds, or a touch log the caller could not read, are rejected before
anything is launched.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import math

import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode_rows_gathered


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _raw_noalloc(ga, plan, batch):
    """The C entry with null buffers: only argument checks can run."""
    return ga.lib.ga_decode_global_hd512_noalloc(
        None, None, None, 0, None, None, None, 1, None, batch, 32, 4, 16, 1, 0.1,
        ga.ctypes.byref(plan), None, None, None)


def test_noalloc_rejects_plan_beyond_scratch(ga):
    """Runs without a GPU: the size check comes before any CUDA call."""
    wl = W.config(5)
    # 256-token chunks: ~200 MB of partials, well past the scratch array
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=32, num_kv_heads=4, head_dim=512,
                             window=0, num_sms=152, fixed_chunk_tokens=256)
    assert plan.workspace_bytes > ga.NOALLOC_SCRATCH_BYTES
    assert _raw_noalloc(ga, plan, wl.batch) == ga.GA_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_rejects_touch_log_plan(ga):
    """Runs without a GPU: a touch log would be written where the caller
    cannot read it, so such a plan is refused before any CUDA call."""
    wl = W.config(1)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=4, num_kv_heads=1, head_dim=512,
                             window=0, num_sms=152, requested_splits=2,
                             flags=ga.GA_PLAN_TOUCH_LOG)
    assert 0 < plan.workspace_bytes <= ga.NOALLOC_SCRATCH_BYTES
    assert _raw_noalloc(ga, plan, wl.batch) == ga.GA_ERR_INVALID_ARG


def _two_calls(ga, fi, plan, rows, kv):
    """Two no-alloc calls in a row (the second with new queries), each
    bit-identical to the workspace call and within tolerance of the oracle."""
    fam = fi.family
    scale = 1.0 / math.sqrt(fam.head_dim)
    ws = ga.workspace_for(plan, fi.q.device)
    err = torch.zeros(1, dtype=torch.int32, device=fi.q.device)
    g = torch.Generator(device="cpu").manual_seed(77)
    for call in range(2):
        if call == 1:
            fi.q.copy_(torch.randn(fi.q.shape, generator=g).to(torch.bfloat16))
        ref = ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                        scale=scale, plan=plan, workspace=ws,
                                        k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
        out = torch.full_like(fi.q, float("nan"))
        ga.ga_decode_global_hd512_noalloc(fi.q, fi.k_pool, fi.v_pool, fi.page_table,
                                          fi.seq_lens, scale=scale, plan=plan, out=out,
                                          k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(out, ref), f"no-alloc call {call} differs from the workspace call"
        assert_close(out[rows].float().cpu().numpy(), oracle_decode_rows_gathered(fi, rows),
                     kv_dtype=kv, what=f"no-alloc call {call} vs oracle")


@pytest.mark.gpu
@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_E4M3])
def test_noalloc_matches_workspace_call_twice(ga, kv):
    """12B-shaped global family (bf16 pools, then E4M3 pools on the tensor-core
    kernel), a 4-way split plan."""
    wl = W.config(2)
    fam = W.Family("global", 16, 2, 512, 0, kv)
    fi = W.make_family_inputs(wl, fam, device="cuda", poison=True)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim, window=0,
                             requested_splits=4)
    assert plan.mode != ga.GA_SPLIT_NONE and 0 < plan.workspace_bytes <= ga.NOALLOC_SCRATCH_BYTES
    _two_calls(ga, fi, plan, W.sample_rows(wl.batch, 6), kv)


@pytest.mark.gpu
def test_noalloc_plan_near_scratch_limit(ga):
    """31B-shaped global family with the smallest page-aligned chunk whose
    partials still fit the array: the partials reach its last megabytes."""
    wl = W.config(3)
    fam = wl.global_
    best = None
    for chunk in range(16, 4097, 16):
        p = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                              num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim, window=0,
                              num_sms=ga.num_sms(), fixed_chunk_tokens=chunk)
        if p.workspace_bytes <= ga.NOALLOC_SCRATCH_BYTES:
            best = p
            break
    assert best is not None and best.workspace_bytes > ga.NOALLOC_SCRATCH_BYTES * 0.9
    fi = W.make_family_inputs(wl, fam, device="cuda", poison=True)
    _two_calls(ga, fi, best, W.sample_rows(wl.batch, 4), W.KV_BF16)
    del fi
    torch.cuda.empty_cache()
