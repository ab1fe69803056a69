"""Randomised parity of multi-query decode: seeded shapes (head dim, KV type,
group size, query count S, window, lengths around page / stage / window
edges, split mode, scale, unit kind) against the fp64 oracle.  Even seeds
force the tcgen05 units of 64 columns, odd seeds the column-parallel mma.sync
units (with E4M3 pools both plans run the 8-column tensor-core kernel), so
both kinds see the same distribution of shapes.  The method: the paged
attention of both families with the S queries of a row at its last S
positions, causal inside the chunk ("visible-cx/Gemma-4-31B-CoreAI" model
card, hybrid-pf64/ bundles: prefill chunks; "Gemma 4 31B on vLLM --
operating-point reference", Operating-point recipes, LIGHT: speculative
verify)."""
import math

import numpy as np
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close
from tests.test_gpu_mq import _decode, _inputs, _oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
EDGE = [0, 1, 3, 15, 16, 17, 63, 127, 128, 129, 255, 256, 257, 1023, 1024, 1025]


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([256, 512]))
    kv = int(rng.choice([0, 0, 1]))
    Hkv = int(rng.choice([1, 2, 3]))
    g = int(rng.choice([1, 2, 3, 8]))
    S = int(rng.choice([2, 3, 5, 8, 13, 16, 33, 64]))
    window = int(rng.choice([1, 5, 40, 200, 1024, 1 << 20])) if D == 256 else 0
    B = int(rng.integers(1, 9))
    lens = rng.integers(0, 1400, size=B)
    pick = rng.random(B) < 0.5
    lens[pick] = rng.choice(EDGE, size=int(pick.sum()))
    split = [dict(requested_splits=1), dict(requested_splits=int(rng.integers(2, 6))),
             dict(fixed_chunk_tokens=16 * int(rng.integers(1, 12))), dict()][int(rng.integers(0, 4))]
    scale = float(rng.choice([1.0 / math.sqrt(D), 0.02]))
    fam = W.Family("local" if window else "global", g * Hkv, Hkv, D, window, kv)
    return fam, S, lens.astype(np.int32), split, scale


@pytest.mark.parametrize("seed", range(24))
def test_random_multi_query_shapes(ga, seed):
    fam, S, lens, split, scale = _case(seed)
    fi, q = _inputs(lens, fam, S, seed=seed)
    units = ga.GA_PLAN_TENSOR_CORE_UNITS if seed % 2 == 0 else ga.GA_PLAN_COLUMN_PARALLEL_UNITS
    plan = ga.ga_plan_splits_mq(lens, q_len=S, num_q_heads=fam.num_q_heads,
                                num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                window=fam.window, flags=units, **split)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _decode(ga, fi, q, fam, plan, err, scale=scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    g = fam.num_q_heads // fam.num_kv_heads
    what = (f"seed {seed}: D={fam.head_dim} kv={fam.kv_dtype} g={g} Hkv={fam.num_kv_heads} "
            f"S={S} W={fam.window} B={len(lens)} {split} col_tile={plan.col_tile}")
    got = out.float().cpu().numpy()
    assert_close(got, _oracle(fi, q, fam, scale=scale), kv_dtype=fam.kv_dtype, what=what)
    for b, L in enumerate(lens):
        for i in range(S):
            if L - S + i < 0:
                assert np.all(got[b, :, i] == 0), what
