"""Pins for the oracle's multi-query decode (S query tokens per row, the last S
positions, causal inside the chunk): brute force with an explicit mask, a
library routine with a boolean causal/window mask, a closed form that exposes
every query's window edge, and chunk parity against one-query decodes
("visible-cx/Gemma-4-31B-CoreAI", hybrid-pf64/ bundles: chunked and
token-by-token walks must agree).
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O

from tests.test_oracle_pins import _paged


def _case(seed, *, Hq, Hkv, D, S, lens, P=16, spare=3):
    g = torch.Generator().manual_seed(seed)
    K = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    V = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    q = torch.randn(len(lens), Hq, S, D, generator=g).to(torch.bfloat16)
    total = sum(-(-L // P) for L in lens) + spare
    perm = torch.randperm(total, generator=g).numpy()
    kp, vp, table, sl = _paged(K, V, P, perm=perm, spare=spare)
    return q, kp, vp, table, sl, K, V


@pytest.mark.parametrize("Hq,Hkv,D,window,S,lens", [
    (4, 2, 16, 8, 4, (40, 33, 17)),
    (4, 1, 32, 0, 3, (40, 2, 16)),
    (8, 8, 8, 5, 2, (16, 17, 31)),
    (16, 2, 8, 20, 4, (50, 3, 64)),
    (8, 1, 24, 0, 4, (70, 15, 1)),
    (2, 2, 8, 1, 3, (9, 30, 0)),
])
def test_mq_matches_brute_force(Hq, Hkv, D, window, S, lens):
    q, kp, vp, table, sl, _, _ = _case(11, Hq=Hq, Hkv=Hkv, D=D, S=S, lens=lens)
    kw = dict(num_kv_heads=Hkv, window=window, scale=1.0 / math.sqrt(D))
    o1 = O.decode_mq(q, kp, vp, table, sl, **kw)
    o2 = O.brute_decode_mq(q, kp, vp, table, sl, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)


def test_mq_matches_torch_sdpa_causal_window():
    """Library special case: fp64 SDPA on dense KV, S queries at the last S
    positions, boolean mask (key <= query position) & (position - key < W)."""
    Hq, Hkv, D, S, Wn = 8, 2, 32, 4, 12
    lens = [40, 24, 7]
    q, kp, vp, table, sl, K, V = _case(12, Hq=Hq, Hkv=Hkv, D=D, S=S, lens=lens)
    got = O.decode_mq(q, kp, vp, table, sl, num_kv_heads=Hkv, window=Wn, scale=0.3)
    for b, L in enumerate(lens):
        k = K[b].double().repeat_interleave(Hq // Hkv, dim=0)[None]   # [1, Hq, L, D]
        v = V[b].double().repeat_interleave(Hq // Hkv, dim=0)[None]
        t = torch.arange(L - S, L)[:, None]                            # query positions
        j = torch.arange(L)[None, :]
        mask = ((j <= t) & (t - j < Wn))[None, None]                    # [1, 1, S, L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double()[None], k, v, attn_mask=mask, scale=0.3)[0]    # [Hq, S, D]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_mq_chunk_parity_with_one_query_rows():
    """Query i of an S-token chunk equals a one-query decode of the same row
    cut at length L - S + i + 1, for both families."""
    Hq, Hkv, D, S = 4, 2, 16, 4
    lens = [37, 16, 5, 64]
    q, kp, vp, table, sl, _, _ = _case(13, Hq=Hq, Hkv=Hkv, D=D, S=S, lens=lens)
    for window in (0, 9):
        kw = dict(num_kv_heads=Hkv, window=window, scale=0.25)
        mq = O.decode_mq(q, kp, vp, table, sl, **kw)
        for i in range(S):
            cut = torch.clamp(sl - S + i + 1, min=0).to(torch.int32)
            one = O.decode(q[:, :, i].contiguous(), kp, vp, table, cut, **kw)
            np.testing.assert_array_equal(mq[:, :, i], one)


@pytest.mark.parametrize("L", [1026, 1027, 1024, 2050])
def test_mq_window_edges_closed_form(L):
    """q = 0 gives uniform weights, and v_j = j makes the output the mean key
    position of each query: (lo_i + t_i) / 2 with t_i = L - S + i and
    lo_i = max(0, t_i - W + 1), so each query's own window edge shows."""
    Wn, P, D, S = 1024, 16, 8, 4
    pos = torch.arange(L, dtype=torch.float64)
    K = [torch.zeros(1, L, D, dtype=torch.bfloat16)]
    Vd = torch.zeros(1, L, D, dtype=torch.float64)
    Vd[0, :, 0] = torch.floor(pos / 256)
    Vd[0, :, 1] = pos - 256 * torch.floor(pos / 256)
    kp, vp, table, sl = _paged(K, [Vd.to(torch.bfloat16)], P)
    q = torch.zeros(1, 1, S, D, dtype=torch.bfloat16)
    out = O.decode_mq(q, kp, vp, table, sl, num_kv_heads=1, window=Wn, scale=1.0)
    for i in range(S):
        t = L - S + i
        lo = max(0, t - Wn + 1)
        mean_pos = 256 * out[0, 0, i, 0] + out[0, 0, i, 1]
        assert abs(mean_pos - (lo + t) / 2) < 1e-9


def test_mq_single_query_is_decode():
    q, kp, vp, table, sl, _, _ = _case(14, Hq=8, Hkv=2, D=16, S=1, lens=(30, 17, 1))
    kw = dict(num_kv_heads=2, window=10, scale=0.5)
    np.testing.assert_array_equal(O.decode_mq(q, kp, vp, table, sl, **kw)[:, :, 0],
                                  O.decode(q[:, :, 0].contiguous(), kp, vp, table, sl, **kw))


def test_mq_short_rows_and_first_query_sees_one_key():
    """L < S: queries at negative positions attend nothing (zeros, lse -inf);
    the query at position 0 sees exactly key 0 (output = v_0)."""
    Hq, Hkv, D, S = 2, 1, 8, 4
    q, kp, vp, table, sl, _, V = _case(15, Hq=Hq, Hkv=Hkv, D=D, S=S, lens=(2,))
    out, lse = O.decode_mq(q, kp, vp, table, sl, num_kv_heads=Hkv, window=0, scale=1.0,
                           return_lse=True)
    assert np.all(out[0, :, :2] == 0) and np.all(np.isneginf(lse[0, :, :2]))
    v0 = V[0][0, 0].double().numpy()
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h, 2], v0, rtol=0, atol=1e-15)
