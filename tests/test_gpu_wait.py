"""Bounded waits.  Host side (kvr_stream_wait): a deadline that passes
before the stream's work ends is reported as a timeout, without a fault and
without disturbing later launches; a long enough deadline sees the work
finish.  Device side (kvr_set_wait_limit): with a bound far below a copy's
latency every streaming kernel's wait for its first copy runs out; the call
returns, the status word reports KVR_ST_WAIT_TIMEOUT, and with the default
bound restored the next calls are bit-identical to the ones before."""
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh

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


def test_device_wait_runs_out_then_recovers():
    wl = synth.WORKLOADS[2]
    case = synth.make_case(wl, accept=oracle.accept_single_step(wl.top_k))
    dc = gh.DevCase(case)
    sel, sel_phys, scores = gh.select(dc)
    out = gh.attention(dc, sel_phys)
    torch.cuda.synchronize()
    assert kvr.kvr_get_status() == 0
    kvr.kvr_set_wait_limit(1)                                   # 1 ns: no copy lands that fast
    try:
        gh.select(dc)
        assert kvr.kvr_get_status() & kvr.KVR_ST_WAIT_TIMEOUT   # the scoring kernel gave up and returned
        gh.attention(dc, sel_phys)
        assert kvr.kvr_get_status() & kvr.KVR_ST_WAIT_TIMEOUT   # so did the attention
    finally:
        kvr.kvr_set_wait_limit(0)                               # back to 2 s
    sel2, sel_phys2, scores2 = gh.select(dc)
    out2 = gh.attention(dc, sel_phys2)
    torch.cuda.synchronize()
    assert kvr.kvr_get_status() == 0
    assert torch.equal(sel2, sel) and torch.equal(sel_phys2, sel_phys) and torch.equal(scores2, scores)
    assert torch.equal(out2, out)
