"""Host logic of bench.py that decides what its JSON line claims (no GPU):
the committed DRAM-traffic records apply only to the workload and the
sources they were taken on, and the L2 claim follows the step's reuse
distance."""
import json
import os
import shutil

import pytest

import bench


def _tree(tmp_path):
    """A copy of the decode sources under a scratch root."""
    for rel in bench.DECODE_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_record_needs_its_workload_and_sources(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    rec = {"decode_local_hd256_e4m3": {"workload": "ragged", "source_hash": h,
                                       "bytes_per_launch": 123}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.committed_traffic("decode_local_hd256_e4m3", "ragged") == 123
    assert bench.committed_traffic("decode_local_hd256_e4m3", "31b") is None
    assert bench.committed_traffic("decode_global_hd512", "ragged") is None
    # any edit to a decode source retires the record
    src = root / bench.DECODE_SOURCES[-1]
    src.write_text(src.read_text() + "\n")
    assert bench.kernel_source_hash() != h
    assert bench.committed_traffic("decode_local_hd256_e4m3", "ragged") is None


def test_committed_records_are_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as fh:
        recs = json.load(fh)
    assert recs
    for name, rec in recs.items():
        assert name.split("_e4m3")[0] in ("decode_global_hd512", "decode_local_hd256")
        assert rec["workload"] in bench.WORKLOADS
        assert len(rec["source_hash"]) == 16 and int(rec["source_hash"], 16) >= 0
        assert rec["bytes_per_launch"] > 0
        assert os.path.exists(os.path.join(bench.ROOT, rec["profile"]))


@pytest.mark.parametrize("sizes,flush", [([200e6, 300e6], False), ([60e6, 50e6], True),
                                         ([100e6], True), ([140e6, 1e6], False)])
def test_l2_claim_follows_the_reuse_distance(sizes, flush):
    layers = [{"bytes": int(b)} for b in sizes]
    text = bench.l2_claim(layers)
    assert text.startswith("NOT flushed" if flush else "no flush")
    # a layer repeated in the step is re-read after the layers between its uses
    a, b = {"bytes": int(70e6)}, {"bytes": int(70e6)}
    assert bench.l2_claim([a, b, a, b]).startswith("no flush")
    assert bench.l2_claim([a, a, b, b]).startswith("NOT flushed")
