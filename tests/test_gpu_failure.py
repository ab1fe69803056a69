"""Failure detection on the GPU without a fault: a bounded wait is made to run
out (the GA_PLAN_TEST_WAIT_TIMEOUT hook: CTA 0 of the launch issues no page),
the kernel reports GA_DEVERR_TIMEOUT through the error word and returns, and
the context stays usable for a normal decode."""
import dataclasses
import math
import time

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    "local_bf16": (W.Family("local", 4, 2, 256, 32), 1),
    "global_bf16": (W.Family("global", 16, 2, 512, 0), 1),
    "local_e4m3": (W.Family("local", 4, 2, 256, 32, 1), 1),        # tensor-core kernel, hd256
    "global_e4m3": (W.Family("global", 16, 2, 512, 0, 1), 1),      # tensor-core kernel, hd512
    "local_bf16_5_queries": (W.Family("local", 4, 2, 256, 32), 5),     # column-parallel units
    "global_bf16_4_queries": (W.Family("global", 16, 2, 512, 0), 4),   # tensor-core mq, hd512
    "local_bf16_32_queries": (W.Family("local", 4, 2, 256, 32), 32),   # tensor-core mq, hd256
    "local_e4m3_4_heads": (W.Family("local", 8, 4, 256, 32, 1), 1),   # units of 4 kv heads
}
# extra plan flags per case
FLAGS = {"local_e4m3_4_heads": "GA_PLAN_KV_E4M3"}


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


@pytest.mark.parametrize("case", sorted(CASES))
def test_wait_runs_out_reports_and_context_survives(ga, case):
    fam, S = CASES[case]
    lens = np.array([200, 77, 130, 40], dtype=np.int32)
    alloc = dataclasses.replace(fam, window=fam.window + S - 1 if fam.window else 0)
    fi = W.make_family_inputs(W.Workload("fail", lens, 16, alloc, alloc), alloc, device=DEV,
                              seed=5)
    if S > 1:
        q = torch.randn(len(lens), fam.num_q_heads, S, fam.head_dim,
                        generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).to(DEV)
        fi = dataclasses.replace(fi, q=q)
    kw = dict(num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
              head_dim=fam.head_dim, window=fam.window, q_len=S, requested_splits=2)
    extra = getattr(ga, FLAGS[case]) if case in FLAGS else 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stall = ga.ga_plan_splits(lens, flags=ga.GA_PLAN_TEST_WAIT_TIMEOUT | extra, **kw)
    if extra:                                  # units of 4 kv heads (set explicitly)
        stall.kv_heads_per_unit = 4
    assert stall.grid > 1                      # other CTAs still run
    fi_run = dataclasses.replace(fi, family=fam)
    t0 = time.time()
    run_decode(ga, fi_run, stall, err=err, out=torch.empty_like(fi.q))
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    word = int(err.item())
    assert word & ga.GA_DEVERR_TIMEOUT, hex(word)
    assert ga.ga_check_error_word(word) == ga.GA_ERR_DEVICE_CHECK
    assert elapsed < 30.0
    # the context is intact: the same call without the hook is correct
    err.zero_()
    plan = ga.ga_plan_splits(lens, flags=extra, **kw)
    if extra:
        plan.kv_heads_per_unit = 4
    out = run_decode(ga, fi_run, plan, err=err, out=torch.empty_like(fi.q))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    scale = 1.0 / math.sqrt(fam.head_dim)
    if S == 1:
        ref = oracle_decode(fi_run)
    else:
        ref = O.decode_mq(fi.q.cpu(), fi.k_pool.cpu(), fi.v_pool.cpu(), fi.page_table.cpu(),
                          fi.seq_lens.cpu(), num_kv_heads=fam.num_kv_heads, window=fam.window,
                          scale=scale)
    assert_close(out.float().cpu().numpy(), ref, kv_dtype=fam.kv_dtype, what=case)


@pytest.mark.parametrize("case", ["local_bf16", "global_e4m3", "local_e4m3_4_heads"])
def test_fused_append_wait_runs_out(ga, case):
    """The decode call with the KV append fused in, under the same hook: the
    timeout is reported and the call returns; the same call without the hook
    then appends (again: the token bits are the same) and decodes correctly."""
    fam, _ = CASES[case]
    lens = np.array([200, 77, 130, 40], dtype=np.int32)
    fi = W.make_family_inputs(W.Workload("fail", lens, 16, fam, fam), fam, device=DEV, seed=7)
    extra = getattr(ga, FLAGS[case]) if case in FLAGS else 0
    kw = dict(num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
              head_dim=fam.head_dim, window=fam.window, requested_splits=2)
    fused = ga.ga_decode_local_hd256_append if fam.window else ga.ga_decode_global_hd512_append
    call_kw = dict(scale=1.0 / math.sqrt(fam.head_dim), k_scale=fi.k_scale, v_scale=fi.v_scale)
    if fam.window:
        call_kw["window"] = fam.window
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for flags in (ga.GA_PLAN_TEST_WAIT_TIMEOUT | extra, extra):
        plan = ga.ga_plan_splits(lens, flags=flags, **kw)
        if extra:
            plan.kv_heads_per_unit = 4
        out = torch.empty_like(fi.q)
        err.zero_()
        t0 = time.time()
        fused(fi.k_new, fi.v_new, fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
              plan=plan, workspace=ga.workspace_for(plan, DEV), out=out, err_word=err, **call_kw)
        torch.cuda.synchronize()
        assert time.time() - t0 < 30.0
        word = int(err.item())
        if flags & ga.GA_PLAN_TEST_WAIT_TIMEOUT:
            assert word & ga.GA_DEVERR_TIMEOUT, hex(word)
        else:
            assert word == 0, hex(word)
    assert_close(out.float().cpu().numpy(), oracle_decode(fi), kv_dtype=fam.kv_dtype, what=case)
