"""The 31B-shaped batch (64 rows, L ~ U[8192, 32768], 32 q heads; local 16 kv
heads hd256 W1024, global 4 kv heads hd512) at full size, decoded under every
plan of the split-KV sweep -- fixed counts 1, 2, 4, 8, 16 and the planner's
own choice -- for bf16 and E4M3 pools of both families.  Sampled rows (first,
last and six others, every query head) are compared with the fp64 oracle at
1e-2 / 4e-3 (bf16) and 3e-2 / 1.5e-2 (E4M3, oracle on the stored codes).

The sweep follows "[Model] Gemma 4 M3 31B", Proposed Plan (the split-KV chunk
policy is re-checked once the global head count changes); the E4M3 pools
follow "Gemma 4 31B on vLLM -- operating-point reference", LIGHT recipe (fp8
KV cache for every layer).  These are exactly the launches that the bench's
split sweep times."""
import pytest
import torch

from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode_rows_gathered, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"

SWEEP = [dict(requested_splits=1), dict(requested_splits=2), dict(requested_splits=4),
         dict(requested_splits=8), dict(requested_splits=16), dict()]
CASES = [("local", W.KV_BF16), ("global", W.KV_BF16), ("local", W.KV_E4M3),
         ("global", W.KV_E4M3)]


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


class _OneFamily:
    """Keeps one family's full-size inputs (up to ~10 GB) and its oracle rows
    at a time; a new (family, dtype) frees the previous one first."""

    def __init__(self):
        self.key = None
        self.fi = None
        self.rows = None
        self.ref = None

    def get(self, name, kv):
        if self.key != (name, kv):
            self.fi = self.ref = None
            torch.cuda.empty_cache()
            wl = W.config(3)
            base = wl.local if name == "local" else wl.global_
            fam = W.Family(base.name, base.num_q_heads, base.num_kv_heads, base.head_dim,
                           base.window, kv)
            self.fi = W.make_family_inputs(wl, fam, device=DEV, poison=True,
                                           release_old=(fam.window > 0))
            self.rows = W.sample_rows(wl.batch, 8)
            self.ref = oracle_decode_rows_gathered(self.fi, self.rows)
            self.key = (name, kv)
        return self.fi, self.rows, self.ref

    def drop(self):
        self.fi = self.ref = None
        self.key = None
        torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def inputs():
    cache = _OneFamily()
    yield cache
    cache.drop()


@pytest.mark.parametrize("split", SWEEP, ids=lambda s: f"s{s.get('requested_splits', 'auto')}")
@pytest.mark.parametrize("family,kv", CASES, ids=lambda c: str(c))
def test_31b_split_sweep_vs_oracle(ga, inputs, family, kv, split):
    fi, rows, ref = inputs.get(family, kv)
    fam = fi.family
    plan = ga.ga_plan_splits(fi.seq_lens.cpu().numpy(), num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window, **split)
    if "requested_splits" in split and split["requested_splits"] > 1:
        assert plan.mode == ga.GA_SPLIT_COUNT and plan.splits == split["requested_splits"]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out[rows].float().cpu().numpy(), ref, kv_dtype=kv,
                 what=f"31B {family} kv={kv} {split}")
