"""Shared test helpers: run one decode through the C ABI and compare it with
the oracle on the same tensors."""
import math

import numpy as np
import torch

from oracle import oracle as O

TOL = {0: (1e-2, 4e-3), 1: (3e-2, 1.5e-2)}   # kv dtype -> (max-abs, relative RMS)


def metrics(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_close(got, ref, kv_dtype=0, what="", extra_abs=None):
    tol_abs, tol_rel = TOL[kv_dtype]
    max_abs, rel = metrics(got, ref)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{what}: non-finite output"
    bound = tol_abs if extra_abs is None else tol_abs + extra_abs
    assert max_abs <= bound and rel <= tol_rel, \
        f"{what}: max_abs {max_abs:.3e} (<= {bound:.1e}), rel_rms {rel:.3e} (<= {tol_rel:.1e})"
    return max_abs, rel


def run_decode(ga, fi, plan, *, scale=None, err=None, out=None, workspace=None, stream=None):
    fam = fi.family
    if scale is None:
        scale = 1.0 / math.sqrt(fam.head_dim)
    if workspace is None:
        workspace = ga.workspace_for(plan, fi.q.device)
    kw = dict(scale=scale, plan=plan, workspace=workspace, out=out, k_scale=fi.k_scale,
              v_scale=fi.v_scale, err_word=err, stream=stream)
    if fam.window > 0:
        return ga.ga_decode_local_hd256(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                        window=fam.window, **kw)
    return ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                     **kw)


def oracle_decode(fi, *, scale=None, rows=None, nthreads=0):
    fam = fi.family
    if scale is None:
        scale = 1.0 / math.sqrt(fam.head_dim)
    kp, vp = fi.k_pool.cpu(), fi.v_pool.cpu()
    return O.decode(fi.q.cpu(), kp, vp, fi.page_table.cpu(), fi.seq_lens.cpu(),
                    num_kv_heads=fam.num_kv_heads, window=fam.window, scale=scale,
                    kv_dtype=fam.kv_dtype,
                    k_scale=None if fi.k_scale is None else fi.k_scale.cpu(),
                    v_scale=None if fi.v_scale is None else fi.v_scale.cpu(),
                    rows=rows, nthreads=nthreads)


def oracle_decode_rows_gathered(fi, rows, *, scale=None, nthreads=0):
    """Oracle on a subset of rows without copying the whole pool to the host:
    only the pages those rows reference are gathered (renumbered)."""
    fam = fi.family
    if scale is None:
        scale = 1.0 / math.sqrt(fam.head_dim)
    rows = [int(r) for r in rows]
    table = fi.page_table[rows].cpu().numpy()
    used = np.unique(table[table >= 0])
    remap = np.full(max(int(fi.num_pages), 1), -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    sub_table = np.where(table >= 0, remap[np.maximum(table, 0)], -1).astype(np.int32)
    idx = torch.as_tensor(used, device=fi.k_pool.device)
    kp = fi.k_pool.index_select(0, idx).cpu()
    vp = fi.v_pool.index_select(0, idx).cpu()
    return O.decode(fi.q[rows].cpu(), kp, vp, torch.from_numpy(sub_table),
                    fi.seq_lens[rows].cpu(), num_kv_heads=fam.num_kv_heads, window=fam.window,
                    scale=scale, kv_dtype=fam.kv_dtype,
                    k_scale=None if fi.k_scale is None else fi.k_scale.cpu(),
                    v_scale=None if fi.v_scale is None else fi.v_scale.cpu(),
                    nthreads=nthreads)
