"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on
the same seeded inputs.  Page indexing and page sets are compared bit-exact;
outputs within max-abs 1e-2 / relative RMS 4e-3 (bf16 KV) and 3e-2 / 1.5e-2
(E4M3 KV, oracle on the same stored codes)."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W
from tests.helpers import assert_close, oracle_decode, oracle_decode_rows_gathered, run_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


@pytest.fixture
def err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _plan(ga, fi, **kw):
    fam = fi.family
    return ga.ga_plan_splits(fi.seq_lens.cpu().numpy(), num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window, **kw)


def _fam(Hq, Hkv, D, Wn, kv=0, name=None):
    return W.Family(name or ("local" if Wn > 0 else "global"), Hq, Hkv, D, Wn, kv)


def _inputs(lens, fam, seed=0, **kw):
    wl = W.Workload("t", np.asarray(lens, dtype=np.int32), 16, fam, fam)
    kw.setdefault("poison", True)
    return W.make_family_inputs(wl, fam, device=DEV, seed=seed, **kw)


SPLITS = [dict(requested_splits=1), dict(requested_splits=2), dict(requested_splits=4),
          dict(requested_splits=16), dict(fixed_chunk_tokens=16), dict(fixed_chunk_tokens=48),
          dict()]


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("D,kv", [(256, 0), (512, 0), (256, 1), (512, 1)])
def test_append_bit_exact(ga, err, D, kv):
    fi = _inputs([40, 33, 16, 1, 300], _fam(8, 2, D, 0, kv), seed=1, poison=False)
    pos = (fi.seq_lens - 1).clone()
    pos[3] = -1                                       # inactive row
    ref_k, ref_v = O.kv_append(fi.k_new.cpu(), fi.v_new.cpu(), fi.k_pool.cpu(), fi.v_pool.cpu(),
                               fi.page_table.cpu(), pos.cpu(), kv_dtype=kv,
                               k_scale=None if fi.k_scale is None else fi.k_scale.cpu(),
                               v_scale=None if fi.v_scale is None else fi.v_scale.cpu())
    ga.ga_kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, fi.page_table, pos,
                    k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(O._np(fi.k_pool.cpu()), ref_k)
    np.testing.assert_array_equal(O._np(fi.v_pool.cpu()), ref_v)


def test_append_e4m3_rounding_edges(ga, err):
    """Ties, subnormals, saturation: device cvt vs the oracle's encoder."""
    fam = _fam(2, 1, 256, 0, 1)
    fi = _inputs([5], fam, seed=2, poison=False)
    vals = np.array([O.e4m3_decode(c) for c in range(0x7F)] , dtype=np.float64)
    mids = (vals[1:] + vals[:-1]) / 2
    cand = np.concatenate([vals, mids, -mids, [500.0, -1e4, 2.0 ** -10, 3 * 2.0 ** -10]])
    x = torch.tensor(cand[:256], dtype=torch.float32)
    x = torch.cat([x, torch.zeros(256 - x.numel())]) if x.numel() < 256 else x
    k_new = x.to(torch.bfloat16).view(1, 1, 256).to(DEV)
    v_new = (-x).to(torch.bfloat16).view(1, 1, 256).to(DEV)
    ks = torch.ones(1, device=DEV)
    vs = torch.full((1,), 0.5, device=DEV)
    pos = torch.tensor([4], dtype=torch.int32, device=DEV)
    ref_k, ref_v = O.kv_append(k_new.cpu(), v_new.cpu(), fi.k_pool.cpu(), fi.v_pool.cpu(),
                               fi.page_table.cpu(), pos.cpu(), kv_dtype=1, k_scale=ks.cpu(),
                               v_scale=vs.cpu())
    ga.ga_kv_append(k_new, v_new, fi.k_pool, fi.v_pool, fi.page_table, pos, k_scale=ks,
                    v_scale=vs, err_word=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(O._np(fi.k_pool.cpu()), ref_k)
    np.testing.assert_array_equal(O._np(fi.v_pool.cpu()), ref_v)


def test_append_bad_page_reports(ga, err):
    fi = _inputs([40, 33], _fam(4, 2, 256, 0), seed=3, poison=False)
    before = fi.k_pool.clone()
    table = fi.page_table.clone()
    table[1, 2] = fi.num_pages + 5                   # row 1 appends at 32 -> logical page 2
    pos = fi.seq_lens - 1
    ga.ga_kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, table, pos, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_POSITION
    # row 0 still written, row 1 skipped
    page0 = int(table[0, 39 // 16])
    assert torch.equal(fi.k_pool[page0, :, 39 % 16], fi.k_new[0])
    changed = (fi.k_pool != before).any(dim=(1, 3))
    assert int(changed.sum()) == 1


# ------------------------------------------------------------------ decode, config 1

@pytest.mark.parametrize("split", SPLITS, ids=lambda s: str(s))
@pytest.mark.parametrize("family", ["local", "global"])
def test_tiny_config_all_splits(ga, err, family, split):
    wl = W.config(1)
    fam = wl.local if family == "local" else wl.global_
    fi = W.make_family_inputs(wl, fam, device=DEV, poison=True)
    plan = _plan(ga, fi, **split)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.float().cpu().numpy(), oracle_decode(fi), what=f"{family} {split}")


@pytest.mark.parametrize("Hq,Hkv,D,Wn", [(8, 8, 256, 20), (8, 2, 256, 40), (16, 2, 512, 0),
                                          (16, 1, 512, 0), (32, 2, 256, 1024), (4, 1, 512, 0),
                                          (20, 1, 256, 64)])
@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=3), dict()])
def test_group_sizes(ga, err, Hq, Hkv, D, Wn, split):
    """g = 1, 4, 8, 16 (two head groups), 20 (three, the last partial)."""
    lens = [1, 15, 16, 17, 100, 1023, 1024, 1025, 2100, 0]
    fi = _inputs(lens, _fam(Hq, Hkv, D, Wn), seed=4)
    plan = _plan(ga, fi, **split)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.float().cpu().numpy()
    assert_close(got, oracle_decode(fi), what=f"g={Hq // Hkv} D={D} W={Wn} {split}")
    assert np.all(got[-1] == 0)                    # empty row


# ------------------------------------------------------------------ page sets

@pytest.mark.parametrize("family,split", [("local", dict(requested_splits=1)),
                                          ("local", dict(requested_splits=4)),
                                          ("global", dict(fixed_chunk_tokens=64)),
                                          ("global", dict(requested_splits=1))])
def test_page_sets_bit_exact(ga, err, family, split):
    """The producer's log of physical pages read equals, page for page, the
    oracle's logical window pages mapped through the table: window pruning
    and paged indexing are exact."""
    lens = [40, 33, 1023, 1024, 1025, 2049, 3000, 1, 0]
    fam = _fam(8, 2, 256, 1024) if family == "local" else _fam(8, 2, 512, 0)
    fi = _inputs(lens, fam, seed=5, release_old=(family == "local"))
    plan = _plan(ga, fi, flags=ga.GA_PLAN_TOUCH_LOG, **split)
    ws = ga.workspace_for(plan, DEV)
    _, _, log = ga.workspace_views(plan, ws)
    log.fill_(-1)
    run_decode(ga, fi, plan, err=err, workspace=ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    log = log.cpu().numpy()
    table = fi.page_table.cpu().numpy()
    rc = 0
    for b, L in enumerate(lens):
        first, n = O.logical_pages(L, fam.window, 16)
        want = [int(table[b, p]) for p in range(first, first + n)]
        got = []
        chunks = 0
        while len(got) < len(want) or (n == 0 and chunks == 0):
            row = log[rc]
            got += [int(x) for x in row if x >= 0]
            rc += 1
            chunks += 1
            if n == 0:
                break
        assert got == want, (b, L)
    assert rc == plan.row_chunks


# ------------------------------------------------------------------ invariants

def test_page_permutation_bit_exact(ga, err):
    fam = _fam(16, 2, 512, 0)
    lens = [700, 33, 1500]
    a = _inputs(lens, fam, seed=6, poison=False)
    b = _inputs(lens, fam, seed=6, poison=False, spare_pages=40)
    # same logical KV, different physical placement: copy a's pages into b's slots
    ta, tb = a.page_table.cpu().numpy(), b.page_table.cpu().numpy()
    for r, L in enumerate(lens):
        for p in range(-(-L // 16)):
            b.k_pool[tb[r, p]] = a.k_pool[ta[r, p]]
            b.v_pool[tb[r, p]] = a.v_pool[ta[r, p]]
    b.q.copy_(a.q)
    for split in (dict(requested_splits=1), dict(fixed_chunk_tokens=256)):
        oa = run_decode(ga, a, _plan(ga, a, **split), err=err)
        ob = run_decode(ga, b, _plan(ga, b, **split), err=err)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
    assert int(err.item()) == 0


def test_batch_invariance_bit_exact_fixed_chunk(ga, err):
    """With a fixed chunk size a row's result does not depend on the rest of
    the batch, bit for bit ("[Model] Gemma 4 M3 31B", Acceptance Criteria:
    batch invariance)."""
    fam = _fam(32, 4, 512, 0)
    lens = [3000, 17, 900, 4096, 1]
    fi = _inputs(lens, fam, seed=7, poison=False)
    plan = _plan(ga, fi, fixed_chunk_tokens=512)
    full = run_decode(ga, fi, plan, err=err).clone()
    for rows in ([0], [3, 1], [2, 4, 0]):
        sub = W.FamilyInputs(fam, fi.q[rows].contiguous(), fi.k_pool, fi.v_pool, None, None,
                             fi.page_table[rows].contiguous(), fi.seq_lens[rows].contiguous(),
                             fi.k_new, fi.v_new, fi.num_pages)
        p2 = _plan(ga, sub, fixed_chunk_tokens=512)
        part = run_decode(ga, sub, p2, err=err)
        torch.cuda.synchronize()
        assert torch.equal(part, full[rows])
    assert int(err.item()) == 0


def test_split_count_each_vs_oracle(ga, err):
    wl = W.config(2)
    fi = W.make_family_inputs(wl, wl.global_, device=DEV, poison=True)
    ref = oracle_decode(fi, rows=list(range(8)))
    for s in (1, 2, 4, 8, 16):
        out = run_decode(ga, fi, _plan(ga, fi, requested_splits=s), err=err)
        torch.cuda.synchronize()
        assert_close(out[:8].float().cpu().numpy(), ref, what=f"splits={s}")
    assert int(err.item()) == 0


# ------------------------------------------------------------------ workloads

@pytest.mark.parametrize("family", ["local", "global"])
def test_12b_config_full(ga, err, family):
    """12B-shaped batch, rows 0-2 at 1023 / 1024 / 1025, all rows checked."""
    wl = W.config(2)
    fam = wl.local if family == "local" else wl.global_
    fi = W.make_family_inputs(wl, fam, device=DEV, poison=True)
    out = run_decode(ga, fi, _plan(ga, fi), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.float().cpu().numpy(), oracle_decode(fi), what=f"12B {family}")


@pytest.mark.parametrize("family", ["local", "global"])
def test_31b_config_sampled(ga, err, family):
    """Full-size 31B-shaped batch in the bench's launch configuration (auto
    plan), outputs of sampled rows against the oracle."""
    wl = W.config(3)
    fam = wl.local if family == "local" else wl.global_
    fi = W.make_family_inputs(wl, fam, device=DEV, release_old=(family == "local"))
    out = run_decode(ga, fi, _plan(ga, fi), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = W.sample_rows(wl.batch, 6)
    ref = oracle_decode_rows_gathered(fi, rows)
    assert_close(out[rows].float().cpu().numpy(), ref, what=f"31B {family}")
    del fi
    torch.cuda.empty_cache()


def test_long_context_sampled(ga, err):
    wl = W.config(4)
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, device=DEV, release_old=(fam.window > 0))
        out = run_decode(ga, fi, _plan(ga, fi), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        rows = [0, 3]
        ref = oracle_decode_rows_gathered(fi, rows, nthreads=8)
        assert_close(out[rows].float().cpu().numpy(), ref, what=f"long {fam.name}")
        del fi
        torch.cuda.empty_cache()


def test_ragged_fp8_local_and_bf16_global_sampled(ga, err):
    wl = W.config(5)
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, device=DEV, release_old=(fam.window > 0),
                                  poison=(fam.window > 0))
        out = run_decode(ga, fi, _plan(ga, fi), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        rows = W.sample_rows(wl.batch, 12)
        ref = oracle_decode_rows_gathered(fi, rows)
        assert_close(out[rows].float().cpu().numpy(), ref, kv_dtype=fam.kv_dtype,
                     what=f"ragged {fam.name}")
        del fi
        torch.cuda.empty_cache()


@pytest.mark.parametrize("D", [256, 512])
def test_e4m3_paths_vs_oracle(ga, err, D):
    fam = _fam(16, 2, D, 1024 if D == 256 else 0, kv=1)
    fi = _inputs([1023, 1024, 1025, 40, 2500, 1], fam, seed=8)
    for split in (dict(requested_splits=1), dict(requested_splits=3)):
        out = run_decode(ga, fi, _plan(ga, fi, **split), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.float().cpu().numpy(), oracle_decode(fi), kv_dtype=1,
                     what=f"e4m3 D={D} {split}")


# ------------------------------------------------------------------ continuation

def test_multiple_window_continuation_with_page_reuse(ga, err):
    """Decode loop across 2W and 3W: append, decode, release pages that fall
    out of the window and hand them to the next logical page of another row
    ("[Model] Gemma 4 M3 31B", Acceptance Criteria: window boundaries with
    multiple-window continuation, KV release and reuse)."""
    Wn, P = 1024, 16
    fam = _fam(8, 2, 256, Wn)
    released = set()
    steps = 12
    lens = np.array([2040, 3065], dtype=np.int32)          # crosses 2W and 3W
    fi = _inputs(lens, fam, seed=9, poison=True, release_old=True, stride_pad=2)
    table = fi.page_table.cpu().numpy().copy()
    free = sorted(set(range(fi.num_pages)) - set(int(x) for x in table[table >= 0]))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    reused = 0
    for step in range(steps):
        for b in range(2):
            lp = int(lens[b]) // P                          # page of this step's token
            if table[b, lp] < 0:
                page = free.pop(0)
                reused += page in released
                table[b, lp] = page
        fi.page_table.copy_(torch.from_numpy(table))
        lens += 1
        seq.copy_(torch.from_numpy(lens))
        step_fi = W.FamilyInputs(fam, fi.q, fi.k_pool, fi.v_pool, None, None, fi.page_table,
                                 seq, fi.k_new, fi.v_new, fi.num_pages)
        ga.ga_kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, fi.page_table, seq - 1,
                        err_word=err)
        out = run_decode(ga, step_fi, _plan(ga, step_fi, requested_splits=2), err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out.float().cpu().numpy(), oracle_decode(step_fi), what=f"step {step}")
        # release pages whose every slot is older than the window; reuse them first
        for b in range(2):
            L = int(lens[b])
            for p in range(table.shape[1]):
                if table[b, p] >= 0 and (p + 1) * P <= L - Wn:
                    released.add(int(table[b, p]))
                    free.insert(0, int(table[b, p]))
                    table[b, p] = -1
        fi.k_new.mul_(-1.0)
    assert reused >= 1


# ------------------------------------------------------------------ edges and errors

def test_peaked_softmax_scale_one(ga, err):
    """Gemma's scale = 1.0 convention: a peaked softmax, outputs near single
    V rows.  Bound: tolerance plus half a bf16 ulp of the output value."""
    fam = _fam(32, 4, 512, 0)
    fi = _inputs([500, 1025, 33], fam, seed=10)
    out = run_decode(ga, fi, _plan(ga, fi), err=err, scale=1.0)
    torch.cuda.synchronize()
    ref = oracle_decode(fi, scale=1.0)
    half_ulp = float(np.abs(ref).max()) * 2.0 ** -9
    assert_close(out.float().cpu().numpy(), ref, what="scale 1.0", extra_abs=half_ulp)


@pytest.mark.parametrize("D,window,kv", [(256, 32, 0), (256, 32, 1), (512, 0, 1)])
def test_max_batch_short_rows(ga, err, D, window, kv):
    """2048 rows (the per-call maximum: each CTA keeps the row prefix in
    shared memory), short and empty rows; bf16 and both E4M3 kernels."""
    fam = _fam(8, 8 if D == 256 else 2, D, window, kv=kv)
    lens = (np.arange(2048) % 50).astype(np.int32)
    fi = _inputs(lens, fam, seed=11, poison=False)
    out = run_decode(ga, fi, _plan(ga, fi), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = list(range(0, 2048, 97))
    assert_close(out[rows].float().cpu().numpy(), oracle_decode(fi, rows=rows), kv_dtype=kv,
                 what=f"B=2048 D={D} kv={kv}")


def test_bad_page_id_and_length_report_without_nan(ga, err):
    fam = _fam(8, 2, 512, 0)
    fi = _inputs([100, 50], fam, seed=12, poison=False)
    fi.page_table[0, 2] = -7
    plan = _plan(ga, fi)
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_PAGE_ID
    assert torch.isfinite(out.float()).all()
    err.zero_()
    fi.seq_lens[1] = 10_000                               # beyond pt_stride * 16
    out = run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_SEQ_LEN
    assert torch.all(out[1] == 0)


@pytest.mark.parametrize("split", [dict(requested_splits=1), dict(requested_splits=3)])
def test_nan_in_attended_kv_propagates(ga, err, split):
    """A NaN in an attended K or V row makes that head's output NaN, as in the
    oracle; rows and heads that never see it stay finite and correct."""
    fam = _fam(8, 2, 512, 0)
    fi = _inputs([100, 70, 300], fam, seed=16, poison=False)
    p0 = int(fi.page_table[0, 3])                 # row 0, keys 48..63
    fi.k_pool[p0, 1, 5, 7] = float("nan")         # kv head 1 -> query heads 4..7
    p2 = int(fi.page_table[2, 10])
    fi.v_pool[p2, 0, 2, 100] = float("nan")       # row 2, kv head 0 -> heads 0..3
    out = run_decode(ga, fi, _plan(ga, fi, **split), err=err).float().cpu().numpy()
    torch.cuda.synchronize()
    ref = oracle_decode(fi)
    assert np.array_equal(np.isnan(out), np.isnan(ref))
    assert np.isnan(out[0, 4:8]).all() and np.isnan(out[2, 0:4, 100]).all()
    ok = ~np.isnan(ref)
    assert_close(out[ok], ref[ok], what="finite part")


@pytest.mark.parametrize("D,window,kv", [(512, 0, 0), (512, 0, 1), (256, 1024, 1)])
def test_kv_alias_one_pool(ga, err, D, window, kv):
    """k_pool is v_pool (K == V): the one-fetch kernel matches the two-pool
    kernel on a copy and the oracle with V = K.  The two kernels may split a
    chunk's pages over different numbers of consumer warps, so their merge
    order (and the last bit) can differ; both are held to the oracle's bar.
    (E4M3 pools of either family run the tensor-core kernel, which fetches
    each block once into a slot that serves both products.)"""
    fam = _fam(32 if D == 512 else 16, 4 if D == 512 else 8, D, window, kv=kv)
    fi = _inputs([700, 33, 1500, 1], fam, seed=17)
    fi.v_pool = fi.k_pool
    if kv:
        fi.v_scale = fi.k_scale * 1.5
    for split in (dict(requested_splits=1), dict(fixed_chunk_tokens=128)):
        plan = _plan(ga, fi, **split)
        one = run_decode(ga, fi, plan, err=err).clone()
        two_fi = W.FamilyInputs(fam, fi.q, fi.k_pool, fi.k_pool.clone(), fi.k_scale, fi.v_scale,
                                fi.page_table, fi.seq_lens, fi.k_new, fi.v_new, fi.num_pages)
        two = run_decode(ga, two_fi, plan, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle_decode(fi)
        assert_close(one.float().cpu().numpy(), ref, kv_dtype=kv, what=f"alias kv={kv} {split}")
        assert_close(two.float().cpu().numpy(), ref, kv_dtype=kv, what=f"copy kv={kv} {split}")
        assert np.array_equal(np.isnan(one.float().cpu().numpy()), np.isnan(two.float().cpu().numpy()))


def test_capacity_check(ga, err):
    fam = _fam(8, 2, 512, 0)
    fi = _inputs([100, 50], fam, seed=13, poison=False)
    plan = ga.ga_plan_splits([20, 20], num_q_heads=8, num_kv_heads=2, head_dim=512, window=0,
                             fixed_chunk_tokens=16)
    run_decode(ga, fi, plan, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_CAPACITY


def test_e4m3_large_q_is_exact_enough_and_inf_q_reported(ga, err):
    """E4M3 decode scales q per head, so a large finite q (beyond f16 range)
    still matches the oracle; an infinite q is reported."""
    fam = _fam(8, 2, 256, 64, kv=1)
    fi = _inputs([40, 70], fam, seed=14)
    fi.q[1, 3] *= 3e4                         # |q| up to ~1e5, peaked softmax for head 3
    out = run_decode(ga, fi, _plan(ga, fi), err=err, scale=1e-5)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out.float().cpu().numpy(), oracle_decode(fi, scale=1e-5), kv_dtype=1,
                 what="large q")
    fi.q[0, 5, 7] = float("inf")
    run_decode(ga, fi, _plan(ga, fi), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ga.GA_DEVERR_Q_RANGE


_BIG_BATCH = [int(x) for x in np.random.default_rng(3).integers(0, 400, 700)]


@pytest.mark.parametrize("lens", [[300, 17, 900, 0], _BIG_BATCH], ids=["4_rows", "700_rows"])
def test_combine_kernel_alone(ga, err, lens):
    """GPU combine on random fp32 partials vs the oracle's LSE merge (700 rows:
    the combine takes blocks of several consecutive rows per CTA)."""
    Hq, D = (8, 512) if len(lens) < 100 else (2, 256)
    plan = ga.ga_plan_splits(lens, num_q_heads=Hq, num_kv_heads=2, head_dim=D, window=0,
                             fixed_chunk_tokens=64)
    g = torch.Generator(device="cpu").manual_seed(15)
    po = torch.randn(plan.row_chunks, Hq, D, generator=g)
    pl = torch.randn(plan.row_chunks, Hq, generator=g) * 3
    pl[1, Hq - 1] = -float("inf")
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = torch.zeros(len(lens), Hq, D, dtype=torch.bfloat16, device=DEV)
    ga.ga_splitkv_combine(po.to(DEV), pl.to(DEV), plan, seq, 64, out, err_word=err)
    torch.cuda.synchronize()
    rc = 0
    for b, L in enumerate(lens):
        n = 0 if L == 0 else (L - 1) // 16 + 1
        S = max(1, -(-n // 4))
        for h in range(Hq):
            if S > 1:
                ref, _ = O.combine(po[rc:rc + S, h].double().numpy(), pl[rc:rc + S, h].double().numpy())
                assert_close(out[b, h].float().cpu().numpy(), ref, what=f"combine {b},{h}")
            else:
                assert torch.all(out[b, h] == 0)          # single-chunk rows untouched
        rc += S
