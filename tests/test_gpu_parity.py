"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the
seeded workloads: summaries value-exact, selections bit-exact, attention
within 2e-3 max-abs and 1e-3 relative L2."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh

pytestmark = pytest.mark.gpu

_CACHE = {}


def accepted_case(cid):
    """Workload cid's cache and query, redrawn until every top-k boundary has
    a score margin of at least 1e-3 (so fp32 and fp64 selections agree)."""
    if cid not in _CACHE:
        wl = synth.WORKLOADS[cid]
        case = synth.make_case(wl, accept=oracle.accept_single_step(wl.top_k))
        _CACHE[cid] = (case, gh.DevCase(case), oracle.summaries(case.k_pool, case.page_table))
    return _CACHE[cid]


def small_case(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=32, n_pages=150, top_k=21)
    base.update(kw)
    wl = synth.custom(**base)
    case = synth.make_case(wl, accept=oracle.accept_single_step(wl.top_k))
    return case, gh.DevCase(case)


@pytest.fixture(autouse=True)
def _status_clean():
    kvr.kvr_get_status()
    yield
    assert kvr.kvr_get_status() == 0


# ---------------------------------------------------------------- summaries

@pytest.mark.parametrize("cid", [1, 2, 3])
def test_summaries_value_exact(cid):
    case, dc, (kmin, kmax) = accepted_case(cid)
    s = gh.f64(dc.summaries())                       # [B][H][N][2][D]
    np.testing.assert_array_equal(s[:, :, :, 0], kmin)
    np.testing.assert_array_equal(s[:, :, :, 1], kmax)


# ---------------------------------------------------------------- selection

@pytest.mark.parametrize("cid", [1, 2, 3])
def test_selection_bit_exact_and_scores_within_bound(cid):
    case, dc, summ = accepted_case(cid)
    wl = case.wl
    sel, sel_phys, scores = gh.select(dc)
    s_ref = oracle.scores(case.q, *summ)
    want = oracle.topk(s_ref, wl.top_k)
    np.testing.assert_array_equal(sel.cpu().numpy(), want)
    np.testing.assert_array_equal(sel_phys.cpu().numpy(), np.take_along_axis(
        case.page_table[:, None, :].repeat(wl.n_kv_heads, 1), want, axis=2))
    tol = gh.score_tolerance(case.q, *summ, wl.group)
    err = np.abs(scores.cpu().numpy().astype(np.float64) - s_ref)
    assert np.all(err <= tol), f"worst score error {err.max():.3g} vs bound {tol[err == err.max()][0]:.3g}"


def test_tie_goes_to_lower_page_id():
    """Two pages with bitwise-identical keys straddle the top-k boundary: the
    lower page id is selected, by the oracle and by the GPU."""
    wl = synth.custom(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=128, page_size=16, n_pages=200, top_k=17)
    case = synth.make_case(wl)
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))[0, 0]
    order = np.argsort(-s, kind="stable")
    # a boundary with clear margins on both sides of the tied pair
    k = next(k for k in range(8, 60) if s[order[k - 2]] - s[order[k - 1]] >= 1e-3
             and s[order[k - 1]] - s[order[k]] >= 1e-3)
    kth = order[k - 1]
    low = [p for p in order[k + 5:] if p < kth]
    high = [p for p in order[k + 5:] if p > kth]
    targets = ([low[-1]] if low else []) + ([high[-1]] if high else [])
    assert targets
    for target in targets:
        c2 = synth.Case(**{**case.__dict__, "k_pool": case.k_pool.copy()})
        c2.k_pool[c2.page_table[0, target]] = c2.k_pool[c2.page_table[0, kth]]
        summ = oracle.summaries(c2.k_pool, c2.page_table)
        want = oracle.topk(oracle.scores(c2.q, *summ), k)[0, 0]
        lo, hi = min(kth, target), max(kth, target)
        assert lo in want and hi not in want
        dc = gh.DevCase(c2)
        sel, _, scores = gh.select(dc, top_k=k)
        np.testing.assert_array_equal(sel.cpu().numpy()[0, 0], want)
        sc = scores.cpu().numpy()[0, 0]
        assert sc[kth] == sc[target]


@pytest.mark.parametrize("n_pages", [300, 3000, 5000])
def test_all_scores_equal_selects_lowest_ids(n_pages):
    """Every page holds the same keys, so all scores tie and the selection is
    pages 0 .. k-1 in order (the histogram search ends at once on L == R)."""
    wl = synth.custom(batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=16, n_pages=n_pages, top_k=37)
    case = synth.make_case(wl)
    c2 = synth.Case(**{**case.__dict__, "k_pool": case.k_pool.copy()})
    c2.k_pool[:] = c2.k_pool[c2.page_table[0, 0]]
    summ = oracle.summaries(c2.k_pool, c2.page_table)
    want = oracle.topk(oracle.scores(c2.q, *summ), wl.top_k)
    np.testing.assert_array_equal(want, np.broadcast_to(np.arange(wl.top_k), want.shape))
    sel, sel_phys, _ = gh.select(gh.DevCase(c2))
    np.testing.assert_array_equal(sel.cpu().numpy(), want)
    np.testing.assert_array_equal(sel_phys.cpu().numpy()[0], c2.page_table[0, want[0]])


def test_ties_across_the_warps_of_the_top_k():
    """4000 pages, ranked by one CTA whose warps each hold a contiguous block
    of 256 pages.  Every page holds the keys of the lowest-scoring page
    except ten near the end, which hold those of the highest-scoring one.
    With k = 1100 the selection is the 1090 lowest ids of the tie, which run
    across five blocks, then the ten, last in page order: both counts that a
    block takes from the blocks below it are exercised."""
    wl = synth.custom(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=128, page_size=16, n_pages=4000, top_k=1100)
    case = synth.make_case(wl)
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))[0, 0]
    lo, hi = case.page_table[0, np.argmin(s)], case.page_table[0, np.argmax(s)]
    hot = np.arange(3500, 3510)
    c2 = synth.Case(**{**case.__dict__, "k_pool": case.k_pool.copy()})
    c2.k_pool[:] = case.k_pool[lo]
    c2.k_pool[c2.page_table[0, hot]] = case.k_pool[hi]
    want = oracle.topk(oracle.scores(c2.q, *oracle.summaries(c2.k_pool, c2.page_table)), wl.top_k)
    np.testing.assert_array_equal(want[0, 0], np.concatenate([np.arange(wl.top_k - hot.size), hot]))
    sel, sel_phys, _ = gh.select(gh.DevCase(c2))
    np.testing.assert_array_equal(sel.cpu().numpy(), want)
    np.testing.assert_array_equal(sel_phys.cpu().numpy()[0, 0], c2.page_table[0, want[0, 0]])


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("cid", [1, 2, 3])
def test_attention_on_oracle_selection(cid):
    case, dc, summ = accepted_case(cid)
    wl = case.wl
    sel = oracle.topk(oracle.scores(case.q, *summ), wl.top_k)
    ref = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel)
    phys = np.take_along_axis(case.page_table[:, None, :].repeat(wl.n_kv_heads, 1), sel, axis=2)
    out = gh.attention(dc, torch.from_numpy(np.ascontiguousarray(phys)).cuda())
    gh.assert_attn_close(out.cpu().numpy(), ref)


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_decode_step_end_to_end(cid):
    """Selection and attention chained on the device, against the oracle step."""
    case, dc, summ = accepted_case(cid)
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table,
                                             case.wl.n_kv_heads, case.wl.top_k, summ=summ)
    sel, sel_phys, _ = gh.select(dc)
    out = gh.attention(dc, sel_phys)
    np.testing.assert_array_equal(sel.cpu().numpy(), sel_ref)
    gh.assert_attn_close(out.cpu().numpy(), out_ref)


SHAPES = [
    dict(),                                                   # ragged chunk (150 pages) and split (21 pages)
    dict(page_size=16, n_pages=97, top_k=33),
    dict(page_size=64, n_pages=70, top_k=5),
    dict(n_q_heads=2, n_kv_heads=2, top_k=9),                  # G = 1
    dict(n_q_heads=8, n_kv_heads=4, top_k=12),                 # G = 2
    dict(n_q_heads=16, n_kv_heads=2, top_k=30, n_pages=64),    # G = 8
    dict(top_k=150),                                           # k = N: dense attention
    dict(top_k=1, batch=3),
    dict(n_pages=1, top_k=1, page_size=16),
    dict(channel_scale=True, n_pages=300, top_k=40),
    dict(n_pages=1500, top_k=100, batch=1, page_size=16),      # ragged; top-k 256 threads x 8 keys
    dict(n_pages=3000, top_k=90, batch=1, page_size=16),       # top-k 512 threads x 8 keys
    dict(n_pages=5000, top_k=130, batch=1, page_size=16, n_kv_heads=1),   # top-k 512 x 16
    dict(n_pages=16384, top_k=256, batch=1, page_size=16, n_q_heads=4, n_kv_heads=1),  # most pages: 1024 x 16
]


@pytest.mark.parametrize("kw", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
def test_small_shapes_and_edges(kw):
    case, dc = small_case(**kw)
    wl = case.wl
    summ = oracle.summaries(case.k_pool, case.page_table)
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table,
                                             wl.n_kv_heads, wl.top_k, summ=summ)
    s = gh.f64(dc.summaries())
    np.testing.assert_array_equal(s[:, :, :, 0], summ[0])
    np.testing.assert_array_equal(s[:, :, :, 1], summ[1])
    sel, sel_phys, _ = gh.select(dc)
    np.testing.assert_array_equal(sel.cpu().numpy(), sel_ref)
    out = gh.attention(dc, sel_phys)
    gh.assert_attn_close(out.cpu().numpy(), out_ref)


@pytest.mark.parametrize("kw", [SHAPES[i] for i in (1, 2, 3, 4, 5, 7, 11)],
                         ids=["P16", "P64", "G1", "G2", "G8", "k1", "N3000"])
def test_speculative_steps_device_and_host_buffers(kw):
    """Two speculative steps on one query at the edge shapes: step 0 corrects
    every head (the oracle's decode step), step 1 (cosine 1) reuses every head,
    whose attention starts before the top-k ends.  kvr_speculative_step on
    device buffers and kvr_speculative_step_host on page-locked ones give the
    same bits."""
    case, dc = small_case(**kw)
    wl = case.wl
    B, Hq, H, D, k = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.top_k
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table, H, k)
    q_host = torch.from_numpy(np.ascontiguousarray(case.q).view(np.int16)).pin_memory()
    runs = []
    for host in (False, True):
        q_prev = torch.zeros((B, Hq, D), dtype=torch.int16, device="cuda")
        sel_prev = torch.zeros((B, H, k), dtype=torch.int32, device="cuda")
        st = kvr.kvr_spec_state(q_prev.data_ptr(), sel_prev.data_ptr(), 0)
        corr = torch.empty((B, H), dtype=torch.uint8, device="cuda")
        used = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
        used_phys = torch.empty_like(used)
        ws = gh.workspace(dc.dims, k, kvr.KVR_OP_STEP_HOST if host else kvr.KVR_OP_STEP).fill_(0xA5)
        steps = []
        for t in range(2):
            if host:
                out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32).pin_memory()
                kvr.kvr_speculative_step_host(dc.dims, st, q_host, dc.summaries(), dc.page_table, dc.k_pool,
                                              dc.v_pool, k, 0.8, 0.0, out, corr, None, used, used_phys, ws,
                                              ws.numel())
            else:
                out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
                kvr.kvr_speculative_step(dc.dims, st, dc.q, dc.summaries(), dc.page_table, dc.k_pool, dc.v_pool,
                                         k, 0.8, 0.0, out, corr, None, used, used_phys, ws, ws.numel())
            torch.cuda.synchronize()
            steps.append((out.cpu().clone(), corr.cpu().clone(), used.cpu().clone(), sel_prev.cpu().clone()))
        runs.append(steps)
    for t in range(2):
        for a, b in zip(runs[0][t], runs[1][t]):
            assert torch.equal(a, b), f"step {t}"
        out, corr, used, sel_new = runs[0][t]
        assert bool(corr.all()) == (t == 0) and bool((corr == 0).all()) == (t == 1)
        np.testing.assert_array_equal(used.numpy(), sel_ref)
        np.testing.assert_array_equal(sel_new.numpy(), sel_ref)
        gh.assert_attn_close(out.numpy(), out_ref)


def test_alternating_selections_and_attention_on_one_workspace():
    """Selection and attention for two queries in turn, twelve times on one
    workspace: each run gives the oracle's selection and its query's bits of
    the first run (no kernel reads what an earlier call left)."""
    case, dc, summ = accepted_case(2)
    wl = case.wl
    q_np = [case.q, synth.make_multi_queries(case, 1)[:, 0]]
    qs = [gh.t16(x) for x in q_np]
    want = [oracle.topk(oracle.scores(x, *summ), wl.top_k) for x in q_np]
    ws = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_STEP)
    first = {}
    for rep in range(12):
        i = rep % 2
        sel, sel_phys, _ = gh.select(dc, q=qs[i], ws=ws)
        out = gh.attention(dc, sel_phys, q=qs[i], ws=ws)
        torch.cuda.synchronize()
        if i == 0:  # the accepted query keeps the top-k margins
            np.testing.assert_array_equal(sel.cpu().numpy(), want[0], err_msg=f"run {rep}")
        if i not in first:
            first[i] = (sel.clone(), out.clone())
        else:
            assert torch.equal(sel, first[i][0]) and torch.equal(out, first[i][1]), f"run {rep}"


@pytest.mark.parametrize("cid", [2, 3])
def test_repeated_selections_on_one_workspace_match_the_oracle(cid):
    """Eight selections in a row on one workspace each give the oracle's
    top-k.  The top-k kernel is resident while the scoring kernel before it
    still writes the scores (programmatic dependent launch), so it must read
    them at L2: through the read-only cache, lines of an earlier call's
    scores were served and most repeated selections differed."""
    case, dc, summ = accepted_case(cid)
    wl = case.wl
    want = oracle.topk(oracle.scores(case.q, *summ), wl.top_k)
    ws = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_SELECT)
    for rep in range(8):
        sel, _, _ = gh.select(dc, ws=ws)
        np.testing.assert_array_equal(sel.cpu().numpy(), want, err_msg=f"run {rep}")


@pytest.mark.parametrize("scale", [0.05, 1.0])
def test_explicit_scale(scale):
    """A flatter softmax (0.05) and a nearly one-hot one (1.0: logits with a
    standard deviation near 11, so a few tokens carry almost all the weight
    and most weights underflow to zero), merged across the split workers."""
    case, dc = small_case()
    wl = case.wl
    sel_ref, _, _ = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k)
    ref = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel_ref, scale=scale)
    _, sel_phys, _ = gh.select(dc)
    gh.assert_attn_close(gh.attention(dc, sel_phys, scale=scale).cpu().numpy(), ref)


def test_repeatable_with_junk_filled_workspace():
    """Five runs on poisoned outputs give bitwise-identical results, with the
    workspaces filled with junk bytes and with zeros: no call depends on a
    workspace's earlier contents."""
    case, dc, _ = accepted_case(2)
    first = None
    for fill in (0xA5, 0x00, 0xFF, 0x5A, 0xA5):
        ws_s = gh.workspace(dc.dims, case.wl.top_k, kvr.KVR_OP_SELECT).fill_(fill)
        ws_a = gh.workspace(dc.dims, case.wl.top_k, kvr.KVR_OP_ATTN).fill_(fill)
        sel, sel_phys, sc = gh.select(dc, ws=ws_s)
        out = gh.attention(dc, sel_phys, ws=ws_a)
        cur = (sel.cpu().numpy(), sc.cpu().numpy(), out.cpu().numpy())
        if first is None:
            first = cur
        for x, y in zip(first, cur):
            np.testing.assert_array_equal(x, y)


def test_out_of_range_page_is_skipped_and_reported():
    case, dc = small_case()
    wl = case.wl
    sel_ref, _, _ = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k)
    _, sel_phys, _ = gh.select(dc)
    bad = sel_phys.clone()
    bad[0, 0, 3] = dc.dims.n_phys_pages + 5
    out = gh.attention(dc, bad)
    assert kvr.kvr_get_status() & kvr.KVR_ST_BAD_INDEX
    # the row attends over the remaining pages only
    fewer = np.delete(sel_ref[:1], 3, axis=2)       # unit (0, 0) without its 4th page
    ref = oracle.attention(case.q[:1], case.k_pool, case.v_pool, case.page_table[:1], fewer)
    gh.assert_attn_close(out.cpu().numpy()[0, :wl.group], ref[0, :wl.group])
    # the other units are unaffected
    ref_all = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel_ref)
    gh.assert_attn_close(out.cpu().numpy()[:, wl.group:], ref_all[:, wl.group:])
