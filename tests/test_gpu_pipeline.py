"""Multi-layer decode pipeline (kvr_pipeline_step) through the C ABI.  Each
layer's results equal, bit for bit, the single-layer step it generalises
(kvr_speculative_step, and so the overlapped step too, for an HBM-resident
layer; the recall step for a host-resident one) and the oracle's
speculative trace of that layer; the
working sets end every step in the same state; the stand-in reads exactly
the bytes it is given; the timing marks and a CUDA-graph replay change no
result."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh
from tests.test_gpu_spec import OverlapRun, SpecRun

pytestmark = pytest.mark.gpu

STEPS = 8


@pytest.fixture(autouse=True)
def _status_clean():
    kvr.kvr_get_status()
    yield
    assert kvr.kvr_get_status() == 0


_DATA = {}


# seeds whose traces, at tau = 0.9, have a step where some KV heads are
# corrected and others not (steps 3, 7 and 4): the recall of such a step is
# split between the side and the prefetch stream
SEEDS = (43, 44, 45)


def layer_data(i):
    """Layer i: its own cache and query trace (top-k and |C - tau| margins of
    at least 1e-3 at every step) and the oracle's speculative run."""
    if i not in _DATA:
        wl = synth.custom(name=f"layer{i}", batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16,
                          n_pages=96, top_k=12, steps=STEPS, tau=0.9, n_jumps=2, seed=SEEDS[i])
        case = synth.make_case(wl, accept=oracle.accept_single_step(wl.top_k))
        summ = oracle.summaries(case.k_pool, case.page_table)
        tr = synth.make_trace(wl, case, accept=oracle.accept_trace_step(summ, wl.n_kv_heads, wl.top_k, wl.tau))
        ref = oracle.speculative_trace(tr.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads,
                                       wl.top_k, wl.tau, summ=summ)
        c = ref["corrected"].reshape(STEPS, -1)
        assert any(c[t].any() and not c[t].all() for t in range(1, STEPS))
        _DATA[i] = (wl, case, gh.DevCase(case), gh.t16(tr.q), ref)
    return _DATA[i]


def _events(n):
    evs = [torch.cuda.Event() for _ in range(n)]
    for e in evs:
        e.record()                       # torch creates the CUDA event on first record
    return evs


class HostCache:
    """Page-locked head-major copy of a layer's cache (shared, read-only)."""

    def __init__(self, case):
        kh, vh = synth.host_hnd(case)
        self.k_host = torch.from_numpy(kh.view(np.int16)).pin_memory()
        self.v_host = torch.from_numpy(vh.view(np.int16)).pin_memory()
        self.host = kvr.kvr_host_kv(self.k_host.data_ptr(), self.v_host.data_ptr())


class HostRun(SpecRun):
    """State, working set and outputs of a host-resident layer."""

    def __init__(self, wl, dc, cache):
        super().__init__(wl, dc)
        B, H, D, P, N, k = wl.batch, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.n_pages, wl.top_k
        S = 2 * k
        self.cache = cache
        self.k_slots = torch.zeros((B, S, P, H, D), dtype=torch.int16, device="cuda")
        self.v_slots = torch.zeros_like(self.k_slots)
        self.p2s = torch.empty((B, H, N), dtype=torch.int32, device="cuda")
        self.s2p = torch.empty((B, H, S), dtype=torch.int32, device="cuda")
        self.wset = kvr.kvr_working_set(self.k_slots.data_ptr(), self.v_slots.data_ptr(), self.p2s.data_ptr(),
                                        self.s2p.data_ptr(), S)
        kvr.kvr_working_set_reset(dc.dims, self.wset)
        self.slot = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
        self.n_copied = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.side = torch.cuda.Stream()
        self.ev_s, self.ev_r = _events(2)

    def step(self, q_t):
        wl, dc = self.wl, self.dc
        self.out.fill_(float("nan"))
        kvr.kvr_speculative_step_recall(dc.dims, self.st, q_t, dc.summaries(), self.cache.host, self.wset,
                                        wl.top_k, wl.tau, 0.0, self.out, self.corrected, self.cbar, self.sel_used,
                                        self.slot, self.n_copied, self.ws, self.ws.numel(),
                                        torch.cuda.current_stream(), self.side, self.ev_s, self.ev_r)

    def state(self):
        return (self.out, self.corrected, self.cbar, self.sel_used, self.slot, self.q_prev, self.sel_prev,
                self.p2s, self.s2p, self.k_slots, self.v_slots, self.n_copied)


class PipeLayer:
    """One layer of the pipeline: the same buffers as the single-layer runs,
    plus the layer's events."""

    def __init__(self, wl, dc, cache=None):
        self.wl, self.dc = wl, dc
        if cache is None:
            self.run = SpecRun(wl, dc)
            self.idx = self.run.sel_used_phys
            self.ev = _events(2)
        else:
            self.run = HostRun(wl, dc, cache)
            self.idx = self.run.slot
            self.ev = _events(3)

    def io(self, q_t):
        r, dc = self.run, self.dc
        if isinstance(r, HostRun):
            return kvr.layer(r.st, q_t, dc.summaries(), r.out, r.corrected, r.cbar, r.sel_used, self.idx, r.ws,
                             r.ws.numel(), self.ev, host=r.cache.host, wset=r.wset, n_copied_opt=r.n_copied)
        return kvr.layer(r.st, q_t, dc.summaries(), r.out, r.corrected, r.cbar, r.sel_used, self.idx, r.ws,
                         r.ws.numel(), self.ev, page_table=dc.page_table, k_pool=dc.k_pool, v_pool=dc.v_pool)

    def state(self):
        r = self.run
        if isinstance(r, HostRun):
            return r.state()
        return (r.out, r.corrected, r.cbar, r.sel_used, r.sel_used_phys, r.q_prev, r.sel_prev)


class Pipeline:
    def __init__(self, specs, compute=None):
        """specs: [(layer id, host-resident?)]."""
        self.layers, self.qs = [], []
        self.caches = {}
        for i, host in specs:
            wl, case, dc, qs, ref = layer_data(i)
            cache = None
            if host:
                if i not in self.caches:
                    self.caches[i] = HostCache(case)
                cache = self.caches[i]
            self.layers.append(PipeLayer(wl, dc, cache))
            self.qs.append(qs)
        self.dims = self.layers[0].dc.dims
        self.side, self.prefetch = torch.cuda.Stream(), torch.cuda.Stream()
        self.compute = compute

    def step(self, t, marks=None, poison=True):
        if poison:
            for L in self.layers:
                L.run.out.fill_(float("nan"))
                L.run.sel_used.fill_(-7)
        wl = self.layers[0].wl
        kvr.kvr_pipeline_step(self.dims, [L.io(q[t]) for L, q in zip(self.layers, self.qs)], self.compute,
                              wl.top_k, wl.tau, 0.0, torch.cuda.current_stream(), self.side, self.prefetch, marks)

    def join(self):
        """Make the current stream wait for every host layer's prefetch."""
        for L in self.layers:
            if len(L.ev) == 3:
                torch.cuda.current_stream().wait_event(L.ev[2])


def _check_oracle(L, ref, t):
    r = L.run
    np.testing.assert_array_equal(r.corrected.cpu().numpy().astype(bool), ref["corrected"][t], err_msg=f"step {t}")
    np.testing.assert_array_equal(r.sel_used.cpu().numpy(), ref["sel_used"][t], err_msg=f"step {t}")
    np.testing.assert_array_equal(r.sel_prev.cpu().numpy(), ref["sel_new"][t], err_msg=f"step {t}")
    gh.assert_attn_close(r.out.cpu().numpy(), ref["out"][t])


def _assert_same(a_state, b_state, what):
    for a, b in zip(a_state, b_state):
        if a.dtype.is_floating_point:
            assert torch.equal(torch.nan_to_num(a, nan=7.0), torch.nan_to_num(b, nan=7.0)), what
        else:
            assert torch.equal(a, b), what


def _word_sum(w: torch.Tensor, lo: int, hi: int) -> int:
    """Sum of the 32-bit words of bytes [lo, hi) of w, modulo 2^32."""
    words = w.view(torch.int32)[lo // 4:hi // 4].to(torch.int64) & 0xFFFFFFFF
    return int(words.sum().item()) % (1 << 32)


def test_hbm_layers_match_overlapped_steps_and_oracle():
    """Three HBM-resident layers with the stand-in between them, eight steps:
    each layer as kvr_speculative_step_overlap alone and as the oracle."""
    qkv, post = 16 * 12345, 16 * ((1 << 20) + 777)        # post long enough for the unrolled loop
    weights = torch.randint(-2**31, 2**31 - 1, ((qkv + post) // 4,), dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    pipe = Pipeline([(0, False), (1, False), (2, False)], kvr.stand_in(weights, qkv, post, sink))
    refs = [OverlapRun(L.wl, L.dc) for L in pipe.layers]
    for t in range(STEPS):
        pipe.step(t)
        for i, (L, R) in enumerate(zip(pipe.layers, refs)):
            R.step(pipe.qs[i][t])
        torch.cuda.synchronize()
        for i, (L, R) in enumerate(zip(pipe.layers, refs)):
            assert L.run.st.step == t + 1
            _assert_same(L.state(), (R.out, R.corrected, R.cbar, R.sel_used, R.sel_used_phys, R.q_prev,
                                     R.sel_prev), f"layer {i} step {t}")
            _check_oracle(L, layer_data(i)[4], t)
    want = 3 * STEPS * (_word_sum(weights, 0, qkv) + _word_sum(weights, qkv, qkv + post)) % (1 << 32)
    assert int(sink.item()) & 0xFFFFFFFF == want


def test_host_layers_match_recall_steps_and_oracle():
    """Two host-resident layers: outputs, slots, maps and copy counts equal
    kvr_speculative_step_recall's, layer by layer, at every step."""
    pipe = Pipeline([(0, True), (1, True)])
    refs = [HostRun(L.wl, L.dc, L.run.cache) for L in pipe.layers]
    for t in range(STEPS):
        pipe.step(t)
        for i, R in enumerate(refs):
            R.step(pipe.qs[i][t])
        torch.cuda.synchronize()
        for i, (L, R) in enumerate(zip(pipe.layers, refs)):
            assert L.run.st.step == t + 1
            _assert_same(L.state(), R.state(), f"layer {i} step {t}")
            _check_oracle(L, layer_data(i)[4], t)
            if t == 0:
                wl = L.wl
                assert int(L.run.n_copied.item()) == wl.batch * wl.n_kv_heads * wl.top_k


def test_mixed_layers_with_marks_and_graph_replay():
    """HBM, host, HBM layers: a run that records the timing marks gives the
    same bits as one without; the marks are in order on each stream; steps
    captured into a CUDA graph and replayed give the eager results."""
    specs = [(0, False), (1, True), (2, False)]
    plain, marked, graphed = Pipeline(specs), Pipeline(specs), Pipeline(specs)
    n = len(specs) * kvr.KVR_PIPE_MARKS
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in marks:
        e.record()
    for t in range(4):
        plain.step(t)
        marked.step(t, marks=marks)
        graphed.step(t)
        torch.cuda.synchronize()
        for L, M in zip(plain.layers, marked.layers):
            _assert_same(L.state(), M.state(), f"marks, step {t}")
        for l, (_, host) in enumerate(specs):
            m = marks[l * kvr.KVR_PIPE_MARKS:(l + 1) * kvr.KVR_PIPE_MARKS]
            # a host layer's side marks follow its selection; an HBM layer
            # records them right after 1 and marks 2-4 right before 5
            order = ((2, 7), (8, 9)) if host else ((1, 7), (8, 9), (10, 2))
            for a, b in ((0, 1), (1, 2), (2, 3), (3, 4), (4, 5), (5, 6), (7, 8), (9, 10), (8, 4)) + order:
                assert m[a].elapsed_time(m[b]) >= -1e-3, (l, a, b)       # ms; timer granularity
            if l + 1 < len(specs):
                assert m[6].elapsed_time(marks[(l + 1) * kvr.KVR_PIPE_MARKS]) >= -1e-3
    # steps 4..7 captured once (the host layer's cross-step event gets a
    # record inside the capture first; its prefetch is joined at the end)
    torch.cuda.synchronize()
    snap = [[x.clone() for x in L.state()] for L in graphed.layers]
    steps0 = [L.run.st.step for L in graphed.layers]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):   # as the recall step's capture
        for L in graphed.layers:
            if len(L.ev) == 3:
                L.ev[2].record()
        for t in range(4, STEPS):
            graphed.step(t, poison=False)
        graphed.join()
    # capture ran nothing: put the state back, then replay
    for L, saved, s0 in zip(graphed.layers, snap, steps0):
        for x, y in zip(L.state(), saved):
            x.copy_(y)
        L.run.st.step = s0
    g.replay()
    for t in range(4, STEPS):
        plain.step(t, poison=False)
    plain.join()
    torch.cuda.synchronize()
    for i, (L, M) in enumerate(zip(plain.layers, graphed.layers)):
        _assert_same(L.state(), M.state(), f"graph, layer {i}")
        _check_oracle(M, layer_data(specs[i][0])[4], STEPS - 1)
