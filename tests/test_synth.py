"""The seeded generator: determinism, layout, bf16 rounding, planted pages,
margins and the speculative query trace's fidelity to the pages.  CPU only."""
import json
import os

import numpy as np
import torch

import oracle
from kv_cache_page_build_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_rounding_matches_torch_on_float32_values():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32).astype(np.float64)
    x[:4] = [0.0, 1.0, -3.5, 1.00390625]                   # includes an exact tie (1 + 2^-8)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(synth.f64_to_bf16_bits(x), want)
    np.testing.assert_array_equal(synth.bf16_bits_to_f64(want),
                                  torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_case_is_deterministic_and_table_is_a_permutation():
    wl = synth.custom(batch=3, n_q_heads=4, n_kv_heads=2, head_dim=16, page_size=4, n_pages=10, top_k=3,
                      n_planted=2, channel_scale=True)
    a, b = synth.make_case(wl), synth.make_case(wl)
    for x, y in [(a.k_pool, b.k_pool), (a.v_pool, b.v_pool), (a.page_table, b.page_table), (a.q, b.q)]:
        np.testing.assert_array_equal(x, y)
    assert sorted(a.page_table.ravel().tolist()) == list(range(wl.batch * wl.n_pages))
    assert not np.array_equal(a.page_table.ravel(), np.arange(wl.batch * wl.n_pages))


def test_host_layout_is_a_pure_rearrangement():
    wl = synth.custom(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=8, page_size=4, n_pages=5, top_k=2)
    case = synth.make_case(wl)
    kh, vh = synth.host_hnd(case)
    for b in range(wl.batch):
        for g in range(wl.n_kv_heads):
            for p in range(wl.n_pages):
                np.testing.assert_array_equal(kh[b, g, p], case.k_pool[case.page_table[b, p], :, g, :])
                np.testing.assert_array_equal(vh[b, g, p], case.v_pool[case.page_table[b, p], :, g, :])


def test_tiny_workload_planted_pages_are_hot_and_margin_holds():
    """Planted pages carry a large share of the exact attention mass; the
    accepted query keeps a 1e-3 score margin at every top-k boundary.  The
    min/max bound ranks these pages low: their keys vary less per channel
    (0.6 sigma around 0.8 q_dir) than an N(0,1) page's, and the bound grows
    with that spread."""
    wl = synth.WORKLOADS[1]
    case = synth.make_case(wl, accept=oracle.accept_single_step(wl.top_k))
    sel, s = oracle.select(case.q, case.k_pool, case.page_table, wl.n_kv_heads, wl.top_k)
    assert np.all(oracle.topk_margin(s, wl.top_k) >= oracle.MARGIN)
    K = synth.bf16_bits_to_f64(case.k_pool)[case.page_table]          # [B][N][P][H][D]
    q = synth.bf16_bits_to_f64(case.q)
    for b in range(wl.batch):
        for h in range(wl.n_q_heads):
            g = h // wl.group
            logit = np.einsum("d,npd->np", q[b, h], K[b, :, :, g]) / np.sqrt(wl.head_dim)
            w = np.exp(logit - logit.max())
            w /= w.sum()
            assert w[case.planted[b, g]].sum() >= 0.25          # 4 of 256 pages
            assert np.all(s[b, g, case.planted[b, g]] < np.median(s[b, g]))


def test_channel_scales_are_log_uniform_in_range():
    wl = synth.custom(batch=1, n_q_heads=8, n_kv_heads=8, head_dim=128, page_size=2, n_pages=2, top_k=1,
                      channel_scale=True)
    ks, vs = synth._channel_scales(wl)
    for s in (ks, vs):
        assert s.min() >= 0.25 and s.max() <= 4.0
        assert abs(np.log(s).mean()) < 0.15          # log-uniform on [ln 1/4, ln 4] has mean 0


def test_speculative_trace_matches_the_pages_observation():
    """Adjacent-step query cosine of 0.84 or more for most steps; the seeded
    topic jumps fall far below the 0.8 threshold."""
    obs = json.load(open(os.path.join(GOLDEN, "query_cosine_observation.json")))
    wl = synth.WORKLOADS[4]
    base = synth.WORKLOADS[2]

    class Head:
        pass
    head = Head()
    head.wl = base
    head.q = np.stack([synth._draw_q(base, b, 0) for b in range(base.batch)])
    tr = synth.make_trace(wl, head)
    assert len(tr.jumps) == wl.n_jumps and tr.q.shape == (wl.steps, base.batch, base.n_q_heads, base.head_dim)
    cb = np.stack([oracle.group_cosine(tr.q[t], tr.q[t - 1], base.n_kv_heads) for t in range(1, wl.steps)])
    jump = np.isin(np.arange(1, wl.steps), tr.jumps)
    assert np.all(cb[jump] < 0.3)
    normal = cb[~jump].ravel()
    assert np.mean(normal >= obs["adjacent_step_cosine_at_least"]) >= 0.75
    assert 0.02 <= np.mean(normal < wl.tau) <= 0.3     # some, not most, heads need correction


def test_trace_rejection_redraws_only_the_rejected_row():
    wl = synth.custom(batch=2, n_q_heads=4, n_kv_heads=2, head_dim=16, page_size=4, n_pages=8, top_k=2,
                      steps=4, tau=0.8)
    case = synth.make_case(wl)
    plain = synth.make_trace(wl, case)
    seen = []

    def reject_first_try_of_row1(t, b, q, qp):
        seen.append((t, b))
        return not (t == 2 and b == 1 and seen.count((2, 1)) == 1)
    tr = synth.make_trace(wl, case, accept=reject_first_try_of_row1)
    np.testing.assert_array_equal(tr.q[:2], plain.q[:2])
    np.testing.assert_array_equal(tr.q[2, 0], plain.q[2, 0])
    assert not np.array_equal(tr.q[2, 1], plain.q[2, 1])
    assert tr.attempts[2, 1] == 1


def test_multi_queries_are_deterministic_and_keep_the_margin():
    """Several queries per step: T AR(1) tokens per sequence from the case's
    query, redrawn until the step's mean page score has a top-k margin of at
    least 1e-3 among the started pages; the same seed gives the same bits."""
    wl = synth.custom(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=32, page_size=8, n_pages=40, top_k=6)
    case = synth.make_case(wl)
    lens = np.array([wl.n_pages * wl.page_size - 3, 17 * wl.page_size + 2], dtype=np.int32)
    summ = oracle.summaries(case.k_pool, case.page_table, seq_len=lens)
    acc = oracle.accept_multi_query(summ, wl.n_kv_heads, wl.top_k, lens, wl.page_size)
    qs = synth.make_multi_queries(case, 4, accept=acc)
    assert qs.shape == (2, 4, 8, 32) and qs.dtype == np.uint16
    np.testing.assert_array_equal(qs, synth.make_multi_queries(case, 4, accept=acc))
    _, s, _ = oracle.multi_query_step(qs, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k,
                                      lens, summ=summ)
    started = oracle.valid_pages(lens, wl.page_size)
    for b in range(wl.batch):
        assert np.all(oracle.topk_margin(s[b, :, :started[b]], wl.top_k) >= 1e-3)
    # the AR(1) run keeps successive tokens close (rho = 0.9)
    x = synth.bf16_bits_to_f64(qs)
    cos = (x[:, 1:] * x[:, :-1]).sum(-1) / np.linalg.norm(x[:, 1:], axis=-1) / np.linalg.norm(x[:, :-1], axis=-1)
    assert cos.mean() > 0.8
