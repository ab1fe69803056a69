"""Algorithmic byte counts (the bench's GB/s numerator) against brute force:
enumerate, for every row, the keys any of its S queries attends (query i at
position L - S + i sees keys j with 0 <= (L - S + i) - j < W, or every j up
to its position in the global family) and the pages holding them, then add q
in, out, the page-table entries, the lengths and the fp8 scales."""
import numpy as np
import pytest

from paged_split_kv_gqa_gb300 import metrics as M


def _brute(lens, *, Hq, Hkv, D, W, S, e, alias=False):
    keys = pages = 0
    for L in lens:
        ks = set()
        for i in range(S):
            p = L - S + i
            if p < 0:
                continue
            lo = max(0, p - W + 1) if W > 0 else 0
            ks.update(range(lo, p + 1))
        keys += len(ks)
        pages += len({k // 16 for k in ks})
    kv = keys * 2 * Hkv * D * e
    if alias:
        kv //= 2
    return kv + 2 * len(lens) * Hq * S * D * 2 + 4 * pages + 4 * len(lens) + (8 * Hkv if e == 1 else 0)


@pytest.mark.parametrize("S", [1, 2, 4, 13])
@pytest.mark.parametrize("W", [0, 1, 5, 40])
@pytest.mark.parametrize("e", [2, 1])
def test_decode_bytes_match_brute_force(S, W, e):
    rng = np.random.default_rng(S * 100 + W + e)
    lens = [0, 1, 3, 15, 16, 17, 33] + [int(x) for x in rng.integers(0, 300, size=6)]
    kw = dict(num_q_heads=8, num_kv_heads=2, head_dim=256, window=W, page_size=16,
              kv_bytes_per_elem=e, q_len=S)
    assert M.decode_bytes(lens, **kw) == _brute(lens, Hq=8, Hkv=2, D=256, W=W, S=S, e=e)
    if W == 0:
        assert M.decode_bytes(lens, kv_alias=True, **kw) == \
            _brute(lens, Hq=8, Hkv=2, D=256, W=W, S=S, e=e, alias=True)
