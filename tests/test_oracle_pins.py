"""Pins for the CPU oracle: each test checks it against something other than
itself -- a library routine, a closed form, brute force, an invariant, or a
value printed on the pages -- so that a dropped term, a wrong sign or index or
a transposed operand anywhere in it fails at least one test.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_split_kv_gqa_gb300 import workloads as W


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _paged(K, V, P, perm=None, spare=0):
    """Pack dense per-row K, V lists ([Hkv, L_b, D] each) into a pool + table."""
    B = len(K)
    Hkv, _, D = K[0].shape
    lens = [k.shape[1] for k in K]
    npg = [-(-L // P) for L in lens]
    total = sum(npg) + spare
    stride = max(max(npg), 1)
    if perm is None:
        perm = np.arange(total)
    kp = torch.zeros(total, Hkv, P, D, dtype=torch.bfloat16)
    vp = torch.zeros(total, Hkv, P, D, dtype=torch.bfloat16)
    table = np.full((B, stride), -1, dtype=np.int32)
    n = 0
    for b in range(B):
        for p in range(npg[b]):
            phys = int(perm[n]); n += 1
            table[b, p] = phys
            lo, hi = p * P, min(lens[b], (p + 1) * P)
            kp[phys, :, : hi - lo] = K[b][:, lo:hi]
            vp[phys, :, : hi - lo] = V[b][:, lo:hi]
    return kp, vp, torch.from_numpy(table), torch.tensor(lens, dtype=torch.int32)


# ------------------------------------------------------------------ numbers

def test_bf16_widening_matches_torch():
    g = torch.Generator().manual_seed(1)
    bits = torch.randint(0, 65536, (4096,), generator=g, dtype=torch.int32)
    bits = torch.cat([bits, torch.tensor([0, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x807F])])
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_bits_to_f64(bits.numpy().astype(np.uint16))
    one = np.array([O.lib().oracle_bf16_to_double(int(b)) for b in bits.numpy()])
    finite = np.isfinite(ref) | np.isinf(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    np.testing.assert_array_equal(one[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([O.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(nan, np.isnan(got))       # 0x7F, 0xFF
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # closed forms from the OCP E4M3 definition
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0xFE) == -448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9 and O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x38) == 1.0 and O.e4m3_decode(0x3C) == 1.5


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(2)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.clamp(-448, 448)
    # every representable value and every midpoint between neighbours
    vals = np.array(sorted(set(O.e4m3_decode(c) for c in range(0x7F) if c != 0x7F)))
    mids = (vals[1:] + vals[:-1]) / 2
    grid = torch.tensor(np.concatenate([vals, mids, -vals, -mids]), dtype=torch.float32)
    x = torch.cat([x, grid])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_closed_forms():
    enc = O.e4m3_encode
    assert enc(1.0) == 0x38
    assert enc(1.0625) == 0x38          # tie between 1.0 and 1.125 -> even mantissa 0
    assert enc(1.1875) == 0x3A          # tie between 1.125 (m=1) and 1.25 (m=2) -> m=2
    assert enc(2.0 ** -10) == 0x00      # tie between 0 and 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02  # tie between m=1 and m=2 subnormals -> 2
    assert enc(-0.0) == 0x80
    assert enc(500.0) == 0x7E and enc(-1e9) == 0xFE      # saturate to finite
    assert enc(float("inf")) == 0x7E and enc(float("-inf")) == 0xFE
    assert enc(float("nan")) == 0x7F
    assert enc(460.0) == 0x7E


# ------------------------------------------------------------------ key sets

@pytest.mark.parametrize("L,Wn,lo", [(40, 32, 8), (33, 32, 1), (32, 32, 0), (1, 32, 0),
                                     (1023, 1024, 0), (1024, 1024, 0), (1025, 1024, 1),
                                     (2049, 1024, 1025), (3073, 1024, 2049), (5, 0, 0)])
def test_key_range_closed_form(L, Wn, lo):
    # query at position L-1 sees j with (L-1) - j < W
    assert O.key_range(L, Wn) == (lo, L)
    brute = [j for j in range(L) if Wn <= 0 or (L - 1) - j < Wn]
    assert (brute[0], brute[-1] + 1) == (lo, L)


@pytest.mark.parametrize("L,Wn,first,count", [
    (40, 32, 0, 3),        # keys [8,40): pages 0:[8,16) 1:[16,32) 2:[32,40)
    (33, 32, 0, 3),        # keys [1,33): pages 0:[1,16) 1 2:[32,33)
    (1023, 1024, 0, 64),   # page 63 holds 15 keys
    (1024, 1024, 0, 64),
    (1025, 1024, 0, 65),   # page 0 [1,16) ... page 64 [1024,1025)
    (2048, 1024, 64, 64),
    (2049, 1024, 64, 65),
    (0, 1024, 0, 0),
])
def test_logical_pages_worked_values(L, Wn, first, count):
    assert O.logical_pages(L, Wn, 16) == (first, count)


def test_logical_pages_brute_force():
    for P in (1, 4, 16):
        for Wn in (0, 1, 5, 16, 32):
            for L in range(0, 80):
                keys = [j for j in range(L) if Wn <= 0 or (L - 1) - j < Wn]
                pages = sorted(set(j // P for j in keys))
                f, n = O.logical_pages(L, Wn, P)
                assert list(range(f, f + n)) == pages, (P, Wn, L)


# ------------------------------------------------------------------ decode

def _rand_case(seed, B=3, Hq=4, Hkv=2, D=16, P=16, lens=(40, 33, 17), kv_dtype=O.KV_BF16):
    wl = W.Workload("t", np.array(lens, dtype=np.int32), P,
                    W.Family("local", Hq, Hkv, D, 0, kv_dtype), W.Family("global", Hq, Hkv, D, 0))
    return W.make_family_inputs(wl, wl.local, seed=seed, spare_pages=4)


@pytest.mark.parametrize("Hq,Hkv,D,window,lens", [
    (4, 2, 16, 32, (40, 33, 17)),
    (4, 1, 32, 0, (40, 33, 1)),
    (8, 8, 8, 5, (16, 17, 31)),
    (16, 2, 8, 20, (50, 3, 64)),
    (8, 1, 24, 0, (70, 15, 16)),
])
def test_decode_matches_brute_force(Hq, Hkv, D, window, lens):
    fi = _rand_case(3, Hq=Hq, Hkv=Hkv, D=D, lens=lens)
    kw = dict(num_kv_heads=Hkv, window=window, scale=1.0 / math.sqrt(D))
    o1 = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    o2 = O.brute_decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)


def test_decode_fp8_matches_brute_force():
    fi = _rand_case(4, Hq=8, Hkv=2, D=32, lens=(45, 16, 3), kv_dtype=O.KV_E4M3)
    # distinct scales per head and per operand, so a swapped scale shows
    k_scale = fi.k_scale * torch.tensor([1.0, 3.0])
    v_scale = fi.v_scale * torch.tensor([0.5, 7.0])
    kw = dict(num_kv_heads=2, window=20, scale=0.2, kv_dtype=O.KV_E4M3,
              k_scale=k_scale, v_scale=v_scale)
    o1 = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    o2 = O.brute_decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    # the stored codes really are e4m3 codes of values in range
    assert fi.k_pool.dtype == torch.uint8


def test_decode_matches_torch_sdpa_fp64():
    """Library special case: fp64 SDPA on dense KV with a boolean window mask;
    GQA by repeat_interleave (consecutive query heads share a kv head)."""
    B, Hq, Hkv, D, P, Wn = 3, 8, 2, 32, 16, 24
    lens = [40, 24, 7]
    g = torch.Generator().manual_seed(5)
    K = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    V = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    q = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16)
    perm = torch.randperm(sum(-(-L // P) for L in lens) + 3, generator=g).numpy()
    kp, vp, table, sl = _paged(K, V, P, perm=perm, spare=3)
    got = O.decode(q, kp, vp, table, sl, num_kv_heads=Hkv, window=Wn, scale=0.3)
    for b, L in enumerate(lens):
        k = K[b].double().repeat_interleave(Hq // Hkv, dim=0)[None]   # [1,Hq,L,D]
        v = V[b].double().repeat_interleave(Hq // Hkv, dim=0)[None]
        pos = torch.arange(L)
        mask = ((L - 1 - pos) < Wn)[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double()[None, :, None, :], k, v, attn_mask=mask, scale=0.3)[0, :, 0]
        np.testing.assert_allclose(got[b], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_hand_worked_two_keys():
    """s = scale*<q,k> = [0, ln 3] -> weights [1/4, 3/4]; o = 4/4 + 3*8/4 = 7."""
    q = _bf16([[[1.0]]])
    K = [_bf16([[[0.0], [1.0]]])]
    V = [_bf16([[[4.0], [8.0]]])]
    kp, vp, table, sl = _paged(K, V, 16)
    out, lse = O.decode(q, kp, vp, table, sl, num_kv_heads=1, window=0, scale=math.log(3.0),
                        return_lse=True)
    assert abs(out[0, 0, 0] - 7.0) < 1e-12
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-12          # ln(e^0 + e^ln3)


@pytest.mark.parametrize("L", [1023, 1024, 1025, 2047, 2048, 2049, 3073])
def test_window_boundaries_closed_form(L):
    """q = 0 gives uniform weights over the window, so with v_j = j the output
    is the mean key position (lo + L - 1) / 2: this exposes the window edge
    at 1023 / 1024 / 1025 and in multiple-window continuation
    ("[Model] Gemma 4 M3 31B", Acceptance Criteria)."""
    Wn, P, D = 1024, 16, 8
    lo = max(0, L - Wn)
    # positions must be exact in bf16: store j as hi*256 + lo8 split over dims
    pos = torch.arange(L, dtype=torch.float64)
    K = [torch.zeros(1, L, D, dtype=torch.bfloat16)]
    Vd = torch.zeros(1, L, D, dtype=torch.float64)
    Vd[0, :, 0] = torch.floor(pos / 256)          # exact integers < 256
    Vd[0, :, 1] = pos - 256 * torch.floor(pos / 256)
    V = [Vd.to(torch.bfloat16)]
    kp, vp, table, sl = _paged(K, V, P)
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    out = O.decode(q, kp, vp, table, sl, num_kv_heads=1, window=Wn, scale=1.0)
    mean_pos = 256 * out[0, 0, 0] + out[0, 0, 1]
    assert abs(mean_pos - (lo + L - 1) / 2) < 1e-9


def test_gqa_block_mapping():
    """kv head c holds v = c + 1 everywhere: query head h must return
    floor(h / g) + 1 (block mapping, not h mod Hkv)."""
    Hq, Hkv, D, P = 8, 4, 8, 16
    L = 20
    g = torch.Generator().manual_seed(6)
    K = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16)]
    V = [(torch.arange(Hkv, dtype=torch.float32) + 1)[:, None, None].expand(Hkv, L, D)
         .to(torch.bfloat16).contiguous()]
    kp, vp, table, sl = _paged(K, V, P)
    q = torch.randn(1, Hq, D, generator=g).to(torch.bfloat16)
    out = O.decode(q, kp, vp, table, sl, num_kv_heads=Hkv, window=0, scale=0.5)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // (Hq // Hkv) + 1, rtol=1e-14)


def test_scale_zero_and_identical_keys_give_mean():
    fi = _rand_case(7, Hq=4, Hkv=2, D=16, lens=(40, 9, 1))
    kw = dict(num_kv_heads=2, window=32)
    o = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, scale=0.0, **kw)
    table, P = fi.page_table.numpy(), 16
    vf = O.bf16_bits_to_f64(O._np(fi.v_pool))
    for b, L in enumerate(fi.seq_lens.tolist()):
        lo = max(0, L - 32)
        for h in range(4):
            vs = np.stack([vf[table[b, j // P], h // 2, j % P] for j in range(lo, L)])
            np.testing.assert_allclose(o[b, h], vs.mean(0), rtol=1e-12, atol=1e-14)


def test_peaked_softmax_selects_argmax_and_is_finite():
    fi = _rand_case(8, Hq=4, Hkv=1, D=64, lens=(60,))
    o = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, num_kv_heads=1,
                 window=0, scale=1e4)
    assert np.isfinite(o).all()
    table, P = fi.page_table.numpy(), 16
    kf = O.bf16_bits_to_f64(O._np(fi.k_pool))
    vf = O.bf16_bits_to_f64(O._np(fi.v_pool))
    qf = O.bf16_bits_to_f64(O._np(fi.q))
    for h in range(4):
        s = [qf[0, h] @ kf[table[0, j // P], 0, j % P] for j in range(60)]
        j = int(np.argmax(s))
        np.testing.assert_allclose(o[0, h], vf[table[0, j // P], 0, j % P], atol=1e-9)


def test_window_at_least_length_equals_global():
    fi = _rand_case(9, lens=(40, 33, 17))
    kw = dict(num_kv_heads=2, scale=0.25)
    a = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, window=40, **kw)
    b = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, window=0, **kw)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ invariants

def test_page_permutation_invariance_exact():
    B, Hkv, D, P = 2, 2, 16, 16
    lens = [70, 33]
    g = torch.Generator().manual_seed(10)
    K = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    V = [torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16) for L in lens]
    q = torch.randn(B, 4, D, generator=g).to(torch.bfloat16)
    n = sum(-(-L // P) for L in lens)
    a = O.decode(q, *_paged(K, V, P), num_kv_heads=Hkv, window=48, scale=0.3)
    perm = torch.randperm(n + 5, generator=g).numpy()
    b = O.decode(q, *_paged(K, V, P, perm=perm, spare=5), num_kv_heads=Hkv, window=48,
                 scale=0.3)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("chunk_pages", [1, 2, 3, 5, 64])
def test_split_count_invariance(chunk_pages):
    fi = _rand_case(11, Hq=8, Hkv=2, D=16, lens=(100, 33, 16, 1))
    kw = dict(num_kv_heads=2, window=70, scale=0.4)
    a, la = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, return_lse=True, **kw)
    b, lb = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                     chunk_pages=chunk_pages, return_lse=True, **kw)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=1e-12)


def test_combine_closed_forms():
    po = np.array([[1.0, 2.0], [3.0, 6.0], [100.0, 100.0]])
    o, lse = O.combine(po, np.array([0.5, 0.5, -np.inf]))
    np.testing.assert_allclose(o, [2.0, 4.0], rtol=1e-15)
    assert abs(lse - (0.5 + math.log(2.0))) < 1e-15
    o, lse = O.combine(po[:2], np.array([0.0, math.log(3.0)]))
    np.testing.assert_allclose(o, [0.25 * 1 + 0.75 * 3, 0.25 * 2 + 0.75 * 6], rtol=1e-14)
    o, lse = O.combine(po[:1], np.array([-np.inf]))
    assert lse == -np.inf and np.all(o == 0)


def test_batch_invariance_exact():
    fi = _rand_case(12, Hq=4, Hkv=2, D=16, lens=(40, 33, 17))
    kw = dict(num_kv_heads=2, window=32, scale=0.3)
    full = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    one = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, rows=[1], **kw)
    np.testing.assert_array_equal(full[1], one[0])
    # other rows' data changed -> row 1 unchanged
    q2 = fi.q.clone(); q2[0] = -q2[0]; q2[2] = 0
    sl2 = fi.seq_lens.clone(); sl2[0] = 5
    other = O.decode(q2, fi.k_pool, fi.v_pool, fi.page_table, sl2, **kw)
    np.testing.assert_array_equal(full[1], other[1])


def test_zero_length_row_is_zero():
    fi = _rand_case(13, lens=(40, 0, 17))
    o = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, num_kv_heads=2,
                 window=0, scale=0.3)
    assert np.all(o[1] == 0) and np.isfinite(o).all()


def test_poisoned_pages_do_not_reach_output():
    """Spare pages, slots past L and slots older than the window hold NaN;
    the definition never reads them, so the output stays finite."""
    wl = W.config(1)
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, poison=True)
        o = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                     num_kv_heads=fam.num_kv_heads, window=fam.window,
                     scale=1 / math.sqrt(fam.head_dim))
        assert np.isfinite(o).all()
        # and the poison is really there
        assert torch.isnan(fi.k_pool.float()).any()


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("kv_dtype", [O.KV_BF16, O.KV_E4M3])
def test_append_roundtrip_through_page_table(kv_dtype):
    wl = W.Workload("t", np.array([40, 33, 16, 1], dtype=np.int32), 16,
                    W.Family("local", 4, 2, 32, 0, kv_dtype), W.Family("global", 4, 2, 32, 0))
    fi = W.make_family_inputs(wl, wl.local, seed=14)
    pos = fi.seq_lens - 1
    pos[2] = -1                       # inactive row: nothing written
    kp, vp = O.kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, fi.page_table, pos,
                         kv_dtype=kv_dtype, k_scale=fi.k_scale, v_scale=fi.v_scale)
    k0, v0 = O._np(fi.k_pool), O._np(fi.v_pool)
    table = fi.page_table.numpy()
    touched = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)   # [page, slot]
    for b, p in enumerate(pos.tolist()):
        if p < 0:
            continue
        page, slot = table[b, p // 16], p % 16
        touched[page, slot] = True
        if kv_dtype == O.KV_BF16:
            np.testing.assert_array_equal(kp[page, :, slot], O._np(fi.k_new)[b])
            np.testing.assert_array_equal(vp[page, :, slot], O._np(fi.v_new)[b])
        else:   # codes equal torch's e4m3 cast of the fp32 quotient (in range here)
            ref_k = (fi.k_new[b].float() / fi.k_scale[:, None]).to(torch.float8_e4m3fn)
            ref_v = (fi.v_new[b].float() / fi.v_scale[:, None]).to(torch.float8_e4m3fn)
            np.testing.assert_array_equal(kp[page, :, slot], ref_k.view(torch.uint8).numpy())
            np.testing.assert_array_equal(vp[page, :, slot], ref_v.view(torch.uint8).numpy())
    # nothing else changed
    mask = ~touched[:, None, :, None] * np.ones_like(kp, dtype=bool)
    np.testing.assert_array_equal(kp[mask], k0[mask])
    np.testing.assert_array_equal(vp[mask], v0[mask])


# ------------------------------------------------------------------ pages' printed values

def test_pages_printed_kv_bytes_per_token(golden_facts):
    """The Core AI card prints 1,966,080 B of fp16 KV per token for the 31B
    (60 layer slots x 16 KV x 512 x K,V x 2 B); the same per-token formula the
    bench uses for algorithmic bytes must reproduce it."""
    f = golden_facts["kv_bytes_per_token_31b_coreai"]
    from paged_split_kv_gqa_gb300 import metrics
    per_layer = metrics.kv_bytes_per_token(f["kv_heads"], f["head_dim"], f["bytes_per_elem"])
    assert per_layer * f["layer_slots"] == f["value"]


@pytest.fixture
def golden_facts():
    import json, os
    with open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")) as fh:
        return json.load(fh)
