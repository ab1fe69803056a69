"""The decode entry point that allocates nothing.

ga_decode_global_hd512_noalloc serves callers that cannot allocate device
memory at decode time (for example a plain-C serving loop without a caching
allocator, where cudaMalloc would synchronise the device mid-step).  Its
split-KV scratch is a device array built into the library.  These tests call
it through the C ABI and check it against ga_decode_global_hd512 given its
own workspace, on two calls in a row; a plan that needs more scratch than the
array holds is rejected before anything is launched.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def test_noalloc_rejects_plan_beyond_scratch(ga):
    """Runs without a GPU: the size check comes before any CUDA call."""
    wl = W.config(5)
    # 256-token chunks: ~200 MB of partials, well past the scratch array
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=32, num_kv_heads=4, head_dim=512,
                             window=0, num_sms=152, fixed_chunk_tokens=256)
    assert plan.workspace_bytes > ga.NOALLOC_SCRATCH_BYTES
    with pytest.raises(ga.GAError) as exc:
        st = ga.lib.ga_decode_global_hd512_noalloc(
            None, None, None, 0, None, None, None, 1, None, wl.batch, 32, 4, 16, 1, 0.1,
            ga.ctypes.byref(plan), None, None, None)
        ga._check(st, "noalloc")
    assert exc.value.status == ga.GA_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice(ga):
    dev = "cuda"
    wl = W.config(2)
    fi = W.make_family_inputs(wl, wl.global_, device=dev, poison=True)
    fam = wl.global_
    scale = 1.0 / math.sqrt(fam.head_dim)
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim, window=0,
                             requested_splits=4)
    assert plan.mode != ga.GA_SPLIT_NONE and 0 < plan.workspace_bytes <= ga.NOALLOC_SCRATCH_BYTES
    ws = ga.workspace_for(plan, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    g = torch.Generator(device="cpu").manual_seed(77)
    for call in range(2):
        if call == 1:                          # second call: new queries, same plan
            fi.q.copy_(torch.randn(fi.q.shape, generator=g).to(torch.bfloat16))
        ref = ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                        scale=scale, plan=plan, workspace=ws, err_word=err)
        out = torch.full_like(fi.q, float("nan"))
        ga.ga_decode_global_hd512_noalloc(fi.q, fi.k_pool, fi.v_pool, fi.page_table,
                                          fi.seq_lens, scale=scale, plan=plan, out=out,
                                          err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64),
                     what=f"no-alloc call {call}")
