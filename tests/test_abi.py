"""The C-ABI library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def _declared():
    text = open(os.path.join(ROOT, "include", "ga.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ga_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("ga_kv_append", "ga_decode_local_hd256", "ga_decode_global_hd512",
              "ga_splitkv_combine", "ga_plan_splits"):
        assert n in names


def test_every_declared_symbol_is_exported(ga):
    lib = ctypes.CDLL(ga._build.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name


def test_python_binding_has_same_names(ga):
    for name in ("ga_kv_append", "ga_decode_local_hd256", "ga_decode_global_hd512",
                 "ga_splitkv_combine", "ga_plan_splits", "ga_check_error_word", "ga_version",
                 "ga_decode_local_hd256_append", "ga_decode_global_hd512_append"):
        assert callable(getattr(ga, name)), name


def test_strerror_and_version(ga):
    assert ga.strerror(0) == "GA_OK"
    assert "WORKSPACE" in ga.strerror(3)
    assert "unknown" in ga.strerror(99)
    assert ga.ga_version() == 0x000400
    assert ga.ga_check_error_word(0) == ga.GA_OK
    assert ga.ga_check_error_word(ga.GA_DEVERR_PAGE_ID) == ga.GA_ERR_DEVICE_CHECK


def test_plan_struct_layout_matches_header(ga, tmp_path):
    """The ctypes mirror of ga_plan against the C compiler's own layout of the
    header's struct (size and every field offset)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [n for n, _ in ga.ga_plan._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"ga.h\"\nint main(void) {\n"
        '  printf("%zu\\n", sizeof(ga_plan));\n'
        + "".join(f'  printf("%zu\\n", offsetof(ga_plan, {n}));\n' for n in names)
        + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(ga.ga_plan)
    assert got[1:] == [getattr(ga.ga_plan, n).offset for n in names]


def test_multi_query_plan(ga):
    """ga_plan_splits_mq: q_len recorded, range checked, partials sized for
    Hq * S columns, pages of the union window of the S queries planned."""
    kw = dict(num_q_heads=4, num_kv_heads=2, head_dim=256, window=32, num_sms=8,
              requested_splits=2)
    one = ga.ga_plan_splits([40, 33], **kw)
    four = ga.ga_plan_splits_mq([40, 33], q_len=4, **kw)
    assert one.q_len == 1 and four.q_len == 4
    assert four.partial_o_offset == one.partial_o_offset == 0
    # partial O: row_chunks x (Hq * S) x D fp32, 256-byte aligned regions
    assert four.partial_lse_offset >= four.row_chunks * 4 * 4 * 256 * 4
    # 4 queries x group 2 = 8 columns: still one head group per kv head
    assert four.units == one.units
    assert one.col_tile == four.col_tile == 8
    # 5 queries x group 2 = 10 columns: one column-parallel unit of 4 tiles of 8
    five = ga.ga_plan_splits_mq([40, 33], q_len=5, **kw)
    assert five.col_tile == 32 and five.units == one.units
    # hd256 below 64 columns: column-parallel units unless tensor-core units
    # are asked for
    eight = ga.ga_plan_splits_mq([40, 33], q_len=8, **kw)           # 16 columns
    assert eight.col_tile == 32 and eight.units == one.units
    eight_tc = ga.ga_plan_splits_mq([40, 33], q_len=8, flags=ga.GA_PLAN_TENSOR_CORE_UNITS, **kw)
    assert eight_tc.col_tile == 64 and eight_tc.units == one.units
    wide = ga.ga_plan_splits_mq([40, 33], q_len=40, **kw)        # 80 columns: 2 units of 64
    assert wide.col_tile == 64 and wide.units == 2 * one.units
    wide_cp = ga.ga_plan_splits_mq([40, 33], q_len=40, flags=ga.GA_PLAN_COLUMN_PARALLEL_UNITS,
                                   **kw)
    assert wide_cp.col_tile == 32 and wide_cp.units == 3 * one.units
    # hd512: tensor-core units from 32 columns (4 queries x group 8)
    g8 = dict(num_q_heads=16, num_kv_heads=2, head_dim=512, window=0, num_sms=8)
    assert ga.ga_plan_splits_mq([40, 33], q_len=2, **g8).col_tile == 32
    assert ga.ga_plan_splits_mq([40, 33], q_len=4, **g8).col_tile == 64
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits_mq([40, 33], q_len=4, flags=ga.GA_PLAN_TENSOR_CORE_UNITS |
                             ga.GA_PLAN_COLUMN_PARALLEL_UNITS, **g8)
    # union window, row of length 33, W = 16: one query reads keys 17..32
    # (pages 1..2); four queries (positions 29..32) read keys 14..32 (pages 0..2)
    w1 = ga.ga_plan_splits([33], num_q_heads=2, num_kv_heads=2, head_dim=256, window=16,
                           num_sms=8, flags=ga.GA_PLAN_TOUCH_LOG)
    w4 = ga.ga_plan_splits_mq([33], q_len=4, num_q_heads=2, num_kv_heads=2, head_dim=256,
                              window=16, num_sms=8, flags=ga.GA_PLAN_TOUCH_LOG)
    assert w1.touch_stride == 2 and w4.touch_stride == 3     # keys 17..32 vs 14..32
    with pytest.raises(ga.GAError):
        ga.ga_plan_splits_mq([40], q_len=0, **kw)
    with pytest.raises(ga.GAError) as e:
        ga.ga_plan_splits_mq([40], q_len=ga.MAX_Q_LEN + 1, **kw)
    assert e.value.status == ga.GA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ host-side rejection
# These calls must return before touching CUDA, so they run without a GPU.

def _plan(ga, **kw):
    args = dict(num_q_heads=4, num_kv_heads=2, head_dim=256, window=32, num_sms=8)
    args.update(kw)
    return ga.ga_plan_splits([40, 33], **args)


FAKE = 0x100000          # aligned fake device addresses: never dereferenced
MIS = 0x100001


def _decode_local(ga, plan, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dt=0, ks=None, vs=None, pt=FAKE, pts=3, sl=FAKE, B=2, Hq=4,
             Hkv=2, W=32, P=16, npg=9, scale=0.0625, ws=None, wsb=0, out=FAKE)
    a.update(over)
    return ga.lib.ga_decode_local_hd256(
        a["q"], a["k"], a["v"], a["dt"], a["ks"], a["vs"], a["pt"], a["pts"], a["sl"], a["B"],
        a["Hq"], a["Hkv"], a["W"], a["P"], a["npg"], a["scale"], ctypes.byref(plan), a["ws"],
        a["wsb"], a["out"], None, None)


def test_decode_rejects_before_launch(ga):
    plan = _plan(ga)
    assert _decode_local(ga, plan, P=8) == ga.GA_ERR_UNSUPPORTED
    assert _decode_local(ga, plan, Hq=3) == ga.GA_ERR_INVALID_ARG          # not a multiple
    assert _decode_local(ga, plan, W=0) == ga.GA_ERR_INVALID_ARG
    assert _decode_local(ga, plan, W=64) == ga.GA_ERR_INVALID_ARG          # plan mismatch
    assert _decode_local(ga, plan, q=MIS) == ga.GA_ERR_INVALID_ARG         # misaligned
    assert _decode_local(ga, plan, out=None) == ga.GA_ERR_INVALID_ARG
    assert _decode_local(ga, plan, dt=7) == ga.GA_ERR_UNSUPPORTED
    assert _decode_local(ga, plan, dt=1) == ga.GA_ERR_INVALID_ARG          # E4M3 needs scales
    assert _decode_local(ga, plan, scale=float("nan")) == ga.GA_ERR_INVALID_ARG
    assert _decode_local(ga, plan, npg=1 << 27) == ga.GA_ERR_UNSUPPORTED   # 2^31 rows
    split = _plan(ga, requested_splits=2)
    assert split.workspace_bytes > 0
    assert _decode_local(ga, split) == ga.GA_ERR_INVALID_ARG               # no workspace
    assert _decode_local(ga, split, ws=FAKE, wsb=split.workspace_bytes - 1) == \
        ga.GA_ERR_WORKSPACE_TOO_SMALL
    assert _decode_local(ga, plan, B=0) == ga.GA_ERR_INVALID_ARG           # plan says B=2
    bad = _plan(ga)
    bad.q_len = 0
    assert _decode_local(ga, bad) == ga.GA_ERR_INVALID_ARG                 # corrupted plan
    bad.q_len = ga.MAX_Q_LEN + 1
    assert _decode_local(ga, bad) == ga.GA_ERR_INVALID_ARG
    bad = _plan(ga)
    bad.col_tile = 16
    assert _decode_local(ga, bad) == ga.GA_ERR_INVALID_ARG
    bad = _plan(ga, requested_splits=2)
    bad.schedule = ga.GA_SCHEDULE_ROWS_BY_SIZE                              # split-count plan
    assert _decode_local(ga, bad, ws=FAKE, wsb=bad.workspace_bytes) == ga.GA_ERR_INVALID_ARG
    big = ga.ga_plan_splits([40] * 597, num_q_heads=4, num_kv_heads=2, head_dim=256, window=32,
                            num_sms=8, fixed_chunk_tokens=16)
    assert big.mode == ga.GA_SPLIT_CHUNK
    big.schedule = ga.GA_SCHEDULE_ROWS_BY_SIZE                   # chunked plan above 596 rows
    assert _decode_local(ga, big, B=597, ws=FAKE, wsb=big.workspace_bytes) == \
        ga.GA_ERR_INVALID_ARG
    bad = _plan(ga)
    bad.schedule = 2                                                        # unknown
    assert _decode_local(ga, bad) == ga.GA_ERR_INVALID_ARG


def test_append_rejects_before_launch(ga):
    f = ga.lib.ga_kv_append
    ok = [FAKE, FAKE, FAKE, FAKE, 0, None, None, FAKE, 3, FAKE, 2, 2, 256, 16, 9, None, None]

    def call(**idx):
        a = list(ok)
        for k, v in idx.items():
            a[int(k[1:])] = v
        return f(*a)

    assert call(a13=8) == ga.GA_ERR_UNSUPPORTED        # page size
    assert call(a12=128) == ga.GA_ERR_UNSUPPORTED      # head dim
    assert call(a4=1) == ga.GA_ERR_INVALID_ARG         # E4M3 without scales
    assert call(a2=MIS) == ga.GA_ERR_INVALID_ARG
    assert call(a0=None) == ga.GA_ERR_INVALID_ARG
    assert call(a10=0) == ga.GA_OK                     # empty batch: nothing to do


def test_combine_rejects_before_launch(ga):
    plan = _plan(ga, requested_splits=2)
    f = ga.lib.ga_splitkv_combine
    assert f(FAKE, FAKE, None, FAKE, 3, FAKE, None, None) == ga.GA_ERR_INVALID_ARG
    assert f(None, FAKE, ctypes.byref(plan), FAKE, 3, FAKE, None, None) == ga.GA_ERR_INVALID_ARG
    assert f(MIS, FAKE, ctypes.byref(plan), FAKE, 3, FAKE, None, None) == ga.GA_ERR_INVALID_ARG
    none = _plan(ga)
    assert f(None, None, ctypes.byref(none), None, 3, None, None, None) == ga.GA_OK


def test_read_stream_rejects_before_launch(ga):
    f = ga.lib.ga_read_stream
    assert f(None, 1 << 20, FAKE, None) == ga.GA_ERR_INVALID_ARG      # no source
    assert f(FAKE, 1 << 20, None, None) == ga.GA_ERR_INVALID_ARG      # no sink
    assert f(MIS, 1 << 20, FAKE, None) == ga.GA_ERR_INVALID_ARG       # unaligned source
    assert f(FAKE, 24, FAKE, None) == ga.GA_ERR_INVALID_ARG           # not a multiple of 16
    assert f(FAKE, 0, FAKE, None) == ga.GA_ERR_INVALID_ARG            # empty


def test_oracle_and_library_share_no_code():
    """The oracle sources never include or import the CUDA path and vice versa."""
    orc = open(os.path.join(ROOT, "oracle", "ga_oracle.c")).read() + \
        open(os.path.join(ROOT, "oracle", "oracle.py")).read()
    assert "ga_geometry" not in orc and "ga_device" not in orc and "import ga" not in orc
    assert "from paged_split_kv_gqa_gb300 import ga" not in orc
    for fn in os.listdir(os.path.join(ROOT, "paged_split_kv_gqa_gb300")):
        if fn.endswith(".py"):
            src = open(os.path.join(ROOT, "paged_split_kv_gqa_gb300", fn)).read()
            assert "oracle" not in src.replace("the oracle", "").replace("oracle's", ""), fn
