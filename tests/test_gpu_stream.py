"""ga_read_stream, the read-ceiling measurement helper: a stream over a
zero buffer runs and leaves the sink untouched; unaligned or odd-sized
buffers are rejected on the host before any launch."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ga():
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga as mod
    return mod


def test_read_stream_runs_and_rejects_bad_buffers(ga):
    buf = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    sink = torch.zeros(1, dtype=torch.int64, device=DEV)
    ga.ga_read_stream(buf, sink)
    ga.ga_read_stream(buf[: 16 * 1001], sink)        # a tail shorter than one grid pass
    torch.cuda.synchronize()
    assert int(sink.item()) == 0                      # fold of zeros is 0, not the trigger
    with pytest.raises(ga.GAError):
        ga.ga_read_stream(buf[1:17], sink)            # unaligned start
    with pytest.raises(ga.GAError):
        ga.ga_read_stream(buf[:24], sink)             # not a multiple of 16 bytes
