"""Bounded host-side wait (kvr_stream_wait): a deadline that passes before
the stream's work ends is reported as a timeout, without a fault and
without disturbing later launches; a long enough deadline sees the work
finish."""
import pytest
import torch

from kv_cache_page_build_b300 import kvr

pytestmark = pytest.mark.gpu


def test_wait_times_out_then_completes():
    w = torch.empty(1 << 29, dtype=torch.int32, device="cuda")        # 2 GiB
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    reads = kvr.stand_in(w, 0, 0, sink)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(20):                                                 # 40 GiB of HBM reads: several ms
        kvr.kvr_stand_in_read(reads, 0, w.numel() * 4, s)
    assert kvr.kvr_stream_wait(s, 0) is False                           # polled once, still running
    assert kvr.kvr_stream_wait(s, 20_000_000) is True                   # 20 s deadline
    assert kvr.kvr_stream_wait(s, 0) is True                            # idle now
    # the "not ready" answers left no error behind for the next launch
    kvr.kvr_stand_in_read(reads, 0, 1 << 20, s)
    assert kvr.kvr_stream_wait(s, 20_000_000) is True
    assert kvr.kvr_get_status(s) == 0
