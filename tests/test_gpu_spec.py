"""Speculative decode (reuse + correction) and streamed recall from a host
cache, through the C ABI, against the oracle's speculative trace."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh
from tests.test_gpu_parity import accepted_case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    kvr.kvr_get_status()
    yield
    assert kvr.kvr_get_status() == 0


_TRACES = {}


def accepted_trace(cid):
    """Workload cid's query trace with both margins (top-k boundary, |C - tau|)
    of at least 1e-3 at every step, and the oracle's speculative run of it."""
    if cid not in _TRACES:
        wl = synth.WORKLOADS[cid]
        case, dc, summ = accepted_case(wl.cache_of)
        tr = synth.make_trace(wl, case, accept=oracle.accept_trace_step(summ, wl.n_kv_heads, wl.top_k, wl.tau))
        ref = oracle.speculative_trace(tr.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads,
                                       wl.top_k, wl.tau, summ=summ)
        _TRACES[cid] = (wl, case, dc, tr, ref)
    return _TRACES[cid]


class SpecRun:
    """Device state and outputs of a speculative run."""

    def __init__(self, wl, dc):
        B, Hq, H, D, k = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.top_k
        self.q_prev = torch.zeros((B, Hq, D), dtype=torch.int16, device="cuda")
        self.sel_prev = torch.zeros((B, H, k), dtype=torch.int32, device="cuda")
        self.st = kvr.kvr_spec_state(self.q_prev.data_ptr(), self.sel_prev.data_ptr(), 0)
        self.out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        self.corrected = torch.empty((B, H), dtype=torch.uint8, device="cuda")
        self.cbar = torch.empty((B, H), dtype=torch.float32, device="cuda")
        self.sel_used = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
        self.sel_used_phys = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
        self.ws = gh.workspace(dc.dims, k, kvr.KVR_OP_STEP)
        self.wl, self.dc = wl, dc

    def step(self, q_t):
        wl, dc = self.wl, self.dc
        self.out.fill_(float("nan"))
        self.sel_used.fill_(-7)
        kvr.kvr_speculative_step(dc.dims, self.st, q_t, dc.summaries(), dc.page_table, dc.k_pool, dc.v_pool,
                                 wl.top_k, wl.tau, 0.0, self.out, self.corrected, self.cbar, self.sel_used,
                                 self.sel_used_phys, self.ws, self.ws.numel())


def test_speculative_trace_matches_oracle():
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    run = SpecRun(wl, dc)
    for t in range(wl.steps):
        run.step(qs[t])
        assert run.st.step == t + 1
        corr = run.corrected.cpu().numpy().astype(bool)
        np.testing.assert_array_equal(corr, ref["corrected"][t], err_msg=f"step {t}")
        np.testing.assert_array_equal(run.sel_used.cpu().numpy(), ref["sel_used"][t], err_msg=f"step {t}")
        np.testing.assert_array_equal(run.sel_prev.cpu().numpy(), ref["sel_new"][t], err_msg=f"step {t}")
        np.testing.assert_array_equal(run.sel_used_phys.cpu().numpy(), np.take_along_axis(
            case.page_table[:, None, :].repeat(wl.n_kv_heads, 1), ref["sel_used"][t], axis=2))
        if t > 0:
            assert np.max(np.abs(run.cbar.cpu().numpy() - ref["cbar"][t])) < 1e-5
        else:
            assert np.all(np.isnan(run.cbar.cpu().numpy()))
        gh.assert_attn_close(run.out.cpu().numpy(), ref["out"][t])
    # the trace exercises both branches of the decision
    assert ref["corrected"][1:].any() and not ref["corrected"][1:].all()
    for t in tr.jumps:
        assert ref["corrected"][t].all()


def test_speculative_step_with_mixed_decisions_matches_oracle():
    """Steps that hold both reused units, whose attention may start before
    the top-k ends, and corrected ones, which wait for it: at each step some
    sequences jump to the trace's query of a distant step (cosine near 0,
    all their KV heads corrected) while the others follow the trace (their
    heads reused).  Every query fed is one the trace accepted (top-k margins
    hold) and every C is far from tau; decisions, selections and outputs
    against the oracle's speculative run of the same sequence."""
    wl, case, dc, tr, _ = accepted_trace(4)
    _, _, summ = accepted_case(wl.cache_of)
    steps = 24
    qs_np = tr.q[:steps].copy()
    for t in range(2, steps):
        for b in range(wl.batch):
            if (t + b) % 3 == 0:
                qs_np[t, b] = tr.q[(t + wl.steps // 2) % wl.steps, b]
    ref = oracle.speculative_trace(qs_np, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads,
                                   wl.top_k, wl.tau, summ=summ)
    mixed = [t for t in range(1, steps) if 0 < ref["corrected"][t].sum() < ref["corrected"][t].size]
    assert len(mixed) >= steps // 2, "the sequence should mix reused and corrected units in most steps"
    assert np.all(np.abs(ref["cbar"][1:] - wl.tau) > 1e-3)
    qs = gh.t16(qs_np)
    run = SpecRun(wl, dc)
    for t in range(steps):
        run.step(qs[t])
        np.testing.assert_array_equal(run.corrected.cpu().numpy().astype(bool), ref["corrected"][t],
                                      err_msg=f"step {t}")
        np.testing.assert_array_equal(run.sel_used.cpu().numpy(), ref["sel_used"][t], err_msg=f"step {t}")
        np.testing.assert_array_equal(run.sel_prev.cpu().numpy(), ref["sel_new"][t], err_msg=f"step {t}")
        gh.assert_attn_close(run.out.cpu().numpy(), ref["out"][t])


def test_speculative_state_checkpoint_resume():
    """Saving (q_prev, sel_prev, step) at step 31 and resuming from it
    reproduces steps 32..63 bit for bit."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    run = SpecRun(wl, dc)
    saved, outs = None, []
    for t in range(wl.steps):
        if t == 32:
            saved = (run.q_prev.clone(), run.sel_prev.clone(), run.st.step)
        run.step(qs[t])
        if t >= 32:
            outs.append((run.out.clone(), run.sel_used.clone(), run.corrected.clone()))
    again = SpecRun(wl, dc)
    again.q_prev.copy_(saved[0])
    again.sel_prev.copy_(saved[1])
    again.st.step = saved[2]
    for i, t in enumerate(range(32, wl.steps)):
        again.step(qs[t])
        for a, b in zip(outs[i], (again.out, again.sel_used, again.corrected)):
            assert torch.equal(a, b), f"step {t}"


def test_speculative_select_alone_matches_step():
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    run = SpecRun(wl, dc)
    ws = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_SELECT)
    for t in range(6):
        kvr.kvr_speculative_select(dc.dims, run.st, qs[t], dc.summaries(), dc.page_table, wl.top_k, wl.tau,
                                   run.corrected, None, run.sel_used, run.sel_used_phys, ws, ws.numel())
        np.testing.assert_array_equal(run.sel_used.cpu().numpy(), ref["sel_used"][t])
        np.testing.assert_array_equal(run.corrected.cpu().numpy().astype(bool), ref["corrected"][t])


class OverlapRun(SpecRun):
    """The same state and outputs, stepped by kvr_speculative_step_overlap
    (decision, then selection on a side stream beside the reused heads'
    attention)."""

    def __init__(self, wl, dc):
        super().__init__(wl, dc)
        self.side = torch.cuda.Stream()
        self.ev_d, self.ev_s = torch.cuda.Event(), torch.cuda.Event()
        self.ev_d.record()                       # torch creates the CUDA event on first record
        self.ev_s.record()

    def step(self, q_t, poison=True):
        wl, dc = self.wl, self.dc
        if poison:
            self.out.fill_(float("nan"))
            self.sel_used.fill_(-7)
        kvr.kvr_speculative_step_overlap(dc.dims, self.st, q_t, dc.summaries(), dc.page_table, dc.k_pool,
                                         dc.v_pool, wl.top_k, wl.tau, 0.0, self.out, self.corrected, self.cbar,
                                         self.sel_used, self.sel_used_phys, self.ws, self.ws.numel(),
                                         torch.cuda.current_stream(), self.side, self.ev_d, self.ev_s)


def test_overlapped_step_matches_oracle_and_sequential_step():
    """Every step of the 64-step trace: the overlapped step gives the oracle's
    decisions and selections, attention within tolerance, and the same bits
    as the sequential kvr_speculative_step."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    ovl, seq = OverlapRun(wl, dc), SpecRun(wl, dc)
    for t in range(wl.steps):
        ovl.step(qs[t])
        seq.step(qs[t])
        torch.cuda.synchronize()
        assert ovl.st.step == t + 1
        np.testing.assert_array_equal(ovl.corrected.cpu().numpy().astype(bool), ref["corrected"][t],
                                      err_msg=f"step {t}")
        np.testing.assert_array_equal(ovl.sel_used.cpu().numpy(), ref["sel_used"][t], err_msg=f"step {t}")
        np.testing.assert_array_equal(ovl.sel_prev.cpu().numpy(), ref["sel_new"][t], err_msg=f"step {t}")
        gh.assert_attn_close(ovl.out.cpu().numpy(), ref["out"][t])
        for a, b in ((ovl.out, seq.out), (ovl.sel_used, seq.sel_used), (ovl.sel_used_phys, seq.sel_used_phys),
                     (ovl.corrected, seq.corrected), (ovl.q_prev, seq.q_prev), (ovl.sel_prev, seq.sel_prev)):
            assert torch.equal(a, b), f"step {t}"
        c_o, c_s = ovl.cbar.cpu().numpy(), seq.cbar.cpu().numpy()
        assert np.array_equal(c_o, c_s, equal_nan=True), f"step {t}"


def test_overlapped_step_replays_from_a_cuda_graph():
    """Steps 8..15 captured into a CUDA graph (the side stream joins the
    capture through the events) and replayed give the eager run's results."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    eager, graph_run = OverlapRun(wl, dc), OverlapRun(wl, dc)
    for t in range(8):
        eager.step(qs[t])
        graph_run.step(qs[t])
    torch.cuda.synchronize()
    snap = (graph_run.q_prev.clone(), graph_run.sel_prev.clone(), graph_run.st.step)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for t in range(8, 16):
            graph_run.step(qs[t], poison=False)
    # capture ran nothing: put the state back, then replay
    graph_run.q_prev.copy_(snap[0])
    graph_run.sel_prev.copy_(snap[1])
    g.replay()
    for t in range(8, 16):
        eager.step(qs[t], poison=False)
    torch.cuda.synchronize()
    for a, b in ((eager.out, graph_run.out), (eager.sel_used, graph_run.sel_used),
                 (eager.sel_prev, graph_run.sel_prev), (eager.q_prev, graph_run.q_prev)):
        assert torch.equal(a, b)
    np.testing.assert_array_equal(eager.sel_used.cpu().numpy(), ref["sel_used"][15])


def test_sequential_step_replays_from_a_cuda_graph():
    """Steps 8..15 of kvr_speculative_step captured into a CUDA graph and
    replayed twice give the bits of an eager run fed the same queries twice:
    a reused unit's attention may start before the top-k ends (its early-start
    word carries the capture's tag), and each replay clears the words it
    used, so the second replay starts as clean as the first."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    eager, graph_run = SpecRun(wl, dc), SpecRun(wl, dc)
    for t in range(8):
        eager.step(qs[t])
        graph_run.step(qs[t])
    torch.cuda.synchronize()
    snap = (graph_run.q_prev.clone(), graph_run.sel_prev.clone())

    def plain(run, q):
        kvr.kvr_speculative_step(dc.dims, run.st, q, dc.summaries(), dc.page_table, dc.k_pool, dc.v_pool,
                                 wl.top_k, wl.tau, 0.0, run.out, run.corrected, run.cbar, run.sel_used,
                                 run.sel_used_phys, run.ws, run.ws.numel())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for t in range(8, 16):
            plain(graph_run, qs[t])
    graph_run.q_prev.copy_(snap[0])  # capture ran nothing
    graph_run.sel_prev.copy_(snap[1])
    for rep in range(2):
        g.replay()
        for t in range(8, 16):
            plain(eager, qs[t])
        torch.cuda.synchronize()
        for a, b in ((eager.out, graph_run.out), (eager.sel_used, graph_run.sel_used),
                     (eager.sel_used_phys, graph_run.sel_used_phys), (eager.corrected, graph_run.corrected),
                     (eager.sel_prev, graph_run.sel_prev), (eager.q_prev, graph_run.q_prev)):
            assert torch.equal(a, b), f"replay {rep}"
        if rep == 0:
            np.testing.assert_array_equal(graph_run.sel_used.cpu().numpy(), ref["sel_used"][15])


@pytest.mark.parametrize("fill", [0xA5, 0xFF])
def test_speculative_trace_does_not_depend_on_workspace_contents(fill):
    """The 64-step trace with the step's workspace refilled with junk bytes
    before every step gives the bits of a run on a zeroed one."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    clean, junk = SpecRun(wl, dc), SpecRun(wl, dc)
    for t in range(wl.steps):
        clean.step(qs[t])
        junk.ws.fill_(fill)
        junk.step(qs[t])
        for a, b in ((clean.out, junk.out), (clean.sel_used, junk.sel_used), (clean.corrected, junk.corrected),
                     (clean.sel_prev, junk.sel_prev)):
            assert torch.equal(a, b), f"step {t}"


def test_host_buffer_step_is_bit_identical_to_the_device_step():
    """kvr_speculative_step_host over the 64-step trace, each query read from
    a row of one page-locked host array (an interior pointer) and the output
    written into alternating page-locked host buffers, with no
    synchronisation between steps: the same bits as kvr_speculative_step on
    device copies, and the oracle's decisions and selections."""
    wl, case, dc, tr, ref = accepted_trace(4)
    qs = gh.t16(tr.q)
    q_host = torch.from_numpy(np.ascontiguousarray(tr.q).view(np.int16)).pin_memory()
    B, Hq, D = wl.batch, wl.n_q_heads, wl.head_dim
    outs = [torch.full((B, Hq, D), float("nan"), dtype=torch.float32).pin_memory() for _ in range(2)]
    host, dev = SpecRun(wl, dc), SpecRun(wl, dc)
    host.ws = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_STEP_HOST)
    assert host.ws.numel() > kvr.kvr_workspace_size(dc.dims, wl.top_k, kvr.KVR_OP_STEP)
    outs_dev = torch.empty((wl.steps, B, Hq, D), dtype=torch.float32, device="cuda")
    used_host = torch.empty((wl.steps, B, wl.n_kv_heads, wl.top_k), dtype=torch.int32, device="cuda")
    evs = [torch.cuda.Event() for _ in range(2)]
    got = []
    for t in range(wl.steps):
        kvr.kvr_speculative_step_host(dc.dims, host.st, q_host[t], dc.summaries(), dc.page_table, dc.k_pool,
                                      dc.v_pool, wl.top_k, wl.tau, 0.0, outs[t & 1], host.corrected, host.cbar,
                                      host.sel_used, host.sel_used_phys, host.ws, host.ws.numel())
        used_host[t].copy_(host.sel_used)
        evs[t & 1].record()
        dev.step(qs[t])
        outs_dev[t].copy_(dev.out)
        if t > 0:  # the previous step's output, once its event has passed
            evs[(t - 1) & 1].synchronize()
            got.append(outs[(t - 1) & 1].clone())
            outs[(t - 1) & 1].fill_(float("nan"))
    torch.cuda.synchronize()
    got.append(outs[(wl.steps - 1) & 1].clone())
    assert host.st.step == wl.steps
    for t in range(wl.steps):
        assert torch.equal(got[t], outs_dev[t].cpu()), f"step {t}"
        np.testing.assert_array_equal(used_host[t].cpu().numpy(), ref["sel_used"][t], err_msg=f"step {t}")
    for a, b in ((host.q_prev, dev.q_prev), (host.sel_prev, dev.sel_prev), (host.corrected, dev.corrected),
                 (host.sel_used_phys, dev.sel_used_phys)):
        assert torch.equal(a, b)


def test_host_buffer_step_rejects_memory_that_is_not_page_locked():
    """Pageable host memory and device memory for q_host or out_host are
    refused before any launch: the state does not advance."""
    wl, case, dc, tr, ref = accepted_trace(4)
    B, Hq, D = wl.batch, wl.n_q_heads, wl.head_dim
    run = SpecRun(wl, dc)
    ws = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_STEP_HOST)
    q_ok = torch.from_numpy(np.ascontiguousarray(tr.q[0]).view(np.int16)).pin_memory()
    out_ok = torch.empty((B, Hq, D), dtype=torch.float32).pin_memory()
    q_pageable = torch.from_numpy(np.ascontiguousarray(tr.q[0]).view(np.int16).copy())
    out_pageable = torch.empty((B, Hq, D), dtype=torch.float32)
    q_device = gh.t16(tr.q[0])
    for q, out in ((q_pageable, out_ok), (q_ok, out_pageable), (q_device, out_ok), (q_ok, run.out)):
        with pytest.raises(kvr.KvrError) as e:
            kvr.kvr_speculative_step_host(dc.dims, run.st, q, dc.summaries(), dc.page_table, dc.k_pool, dc.v_pool,
                                          wl.top_k, wl.tau, 0.0, out, run.corrected, run.cbar, run.sel_used,
                                          run.sel_used_phys, ws, ws.numel())
        assert e.value.code == kvr.KVR_ERR_INVALID_ARG
        assert run.st.step == 0
    kvr.kvr_speculative_step_host(dc.dims, run.st, q_ok, dc.summaries(), dc.page_table, dc.k_pool, dc.v_pool,
                                  wl.top_k, wl.tau, 0.0, out_ok, run.corrected, run.cbar, run.sel_used,
                                  run.sel_used_phys, ws, ws.numel())
    torch.cuda.synchronize()
    assert run.st.step == 1
    assert np.isfinite(out_ok.numpy()).all()


# ---------------------------------------------------------------- host-resident cache

def test_recall_trace_matches_oracle_and_hbm_path():
    wl, case, dc, tr, ref = accepted_trace(5)
    B, Hq, H, D, P, N, k = (wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.page_size, wl.n_pages,
                            wl.top_k)
    S = 2 * k
    kh, vh = synth.host_hnd(case)
    k_host = torch.from_numpy(kh.view(np.int16)).pin_memory()
    v_host = torch.from_numpy(vh.view(np.int16)).pin_memory()
    del kh, vh
    k_slots = torch.zeros((B, S, P, H, D), dtype=torch.int16, device="cuda")
    v_slots = torch.zeros_like(k_slots)
    p2s = torch.empty((B, H, N), dtype=torch.int32, device="cuda")
    s2p = torch.empty((B, H, S), dtype=torch.int32, device="cuda")
    host = kvr.kvr_host_kv(k_host.data_ptr(), v_host.data_ptr())
    wset = kvr.kvr_working_set(k_slots.data_ptr(), v_slots.data_ptr(), p2s.data_ptr(), s2p.data_ptr(), S)
    kvr.kvr_working_set_reset(dc.dims, wset)
    run = SpecRun(wl, dc)
    sel_used_slot = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    n_copied = torch.zeros(1, dtype=torch.int32, device="cuda")
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    ev_s, ev_r = torch.cuda.Event(), torch.cuda.Event()
    ev_s.record()                                  # torch creates the CUDA event on first record
    ev_r.record()
    qs = gh.t16(tr.q)
    ws_a = gh.workspace(dc.dims, k, kvr.KVR_OP_ATTN)
    bidx = torch.arange(B, device="cuda")[:, None, None]
    gidx = torch.arange(H, device="cuda")[None, :, None]
    for t in range(wl.steps):
        run.out.fill_(float("nan"))
        kvr.kvr_speculative_step_recall(dc.dims, run.st, qs[t], dc.summaries(), host, wset, k, wl.tau, 0.0,
                                        run.out, run.corrected, run.cbar, run.sel_used, sel_used_slot, n_copied,
                                        run.ws, run.ws.numel(), main, side, ev_s, ev_r)
        torch.cuda.synchronize()
        if t == 0:
            assert int(n_copied.item()) == B * H * k        # cold start: the whole first selection
        np.testing.assert_array_equal(run.corrected.cpu().numpy().astype(bool), ref["corrected"][t])
        np.testing.assert_array_equal(run.sel_used.cpu().numpy(), ref["sel_used"][t])
        gh.assert_attn_close(run.out.cpu().numpy(), ref["out"][t])
        # the same selection read from the HBM-resident pool gives the same bits
        phys = torch.gather(dc.page_table[:, None, :].expand(B, H, N), 2, run.sel_used.long())
        hbm = gh.attention(dc, phys.contiguous(), q=qs[t], ws=ws_a)
        assert torch.equal(hbm, run.out), f"step {t}"
        # every resident slot holds exactly its page, and maps agree both ways
        s2p_now = s2p.long()
        resident = s2p_now >= 0
        pages = s2p_now.clamp(min=0)
        assert torch.equal(torch.gather(p2s.long(), 2, pages)[resident],
                           torch.arange(S, device="cuda").expand(B, H, S)[resident])
        phys_res = dc.page_table.long()[bidx.squeeze(-1), pages.reshape(B, -1)].reshape(B, H, S)
        want_k = dc.k_pool[phys_res, :, gidx, :]                       # [B][H][S][P][D]
        got_k = k_slots.permute(0, 3, 1, 2, 4)                         # [B][H][S][P][D]
        assert torch.equal(got_k[resident], want_k[resident])
        want_v = dc.v_pool[phys_res, :, gidx, :]
        assert torch.equal(v_slots.permute(0, 3, 1, 2, 4)[resident], want_v[resident])
        # the pages used by this step are resident where sel_used_slot says
        slot_of_used = sel_used_slot.long() - bidx * S
        assert torch.equal(torch.gather(s2p_now, 2, slot_of_used), run.sel_used.long())
