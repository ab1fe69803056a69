"""The decode step captured in a CUDA graph and replayed.

Serving captures the decode step per batch bucket ("[Model] Gemma 4 M3 31B",
Proposed Plan: decode graph bucket set).  The library's calls enqueue only
kernels on the caller's stream with host-encoded parameters, so a captured
step replays with new q, new tokens and longer seq_lens read on the device,
as long as the plan was made for lengths at least as large.
"""
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def test_captured_decode_step_replays(ga):
    dev = "cuda"
    steps = 3
    lens0 = np.array([1020, 1500, 40, 2047], dtype=np.int32)
    fams = [W.Family("local", 16, 8, 256, 1024), W.Family("global", 16, 2, 512, 0)]
    wl = W.Workload("graph", lens0 + steps, 16, fams[0], fams[1])     # room for the new tokens
    state = []
    for fam in fams:
        # no NaN poison here: the poison pattern follows the final lengths, and the
        # first replays attend keys that are older than the final window
        fi = W.make_family_inputs(wl, fam, device=dev, poison=False)
        fi.seq_lens.copy_(torch.from_numpy(lens0))
        upper = lens0 + steps
        plan = ga.ga_plan_splits(upper, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, requested_splits=2)
        state.append(dict(fam=fam, fi=fi, plan=plan, ws=ga.workspace_for(plan, dev),
                          out=torch.zeros_like(fi.q), pos=(fi.seq_lens - 1).contiguous()))
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        for s in state:
            fi, fam = s["fi"], s["fam"]
            ga.ga_kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, fi.page_table, s["pos"],
                            err_word=err)
            kw = dict(scale=1 / math.sqrt(fam.head_dim), plan=s["plan"], workspace=s["ws"],
                      out=s["out"], err_word=err)
            if fam.window:
                ga.ga_decode_local_hd256(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                         window=fam.window, **kw)
            else:
                ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table,
                                          fi.seq_lens, **kw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # first launches set kernel attributes
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = torch.Generator(device="cpu").manual_seed(3)
    for k in range(steps):
        for s in state:                          # next token: new q, new K/V, length + 1
            fi = s["fi"]
            fi.q.copy_(torch.randn(fi.q.shape, generator=g).to(torch.bfloat16))
            fi.k_new.copy_(torch.randn(fi.k_new.shape, generator=g).to(torch.bfloat16))
            fi.v_new.copy_(torch.randn(fi.v_new.shape, generator=g).to(torch.bfloat16))
            fi.seq_lens.add_(1)
            s["pos"].copy_(fi.seq_lens - 1)
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for s in state:
            assert_close(s["out"].float().cpu().numpy(), oracle_decode(s["fi"]),
                         what=f"replay {k} {s['fam'].name}")
