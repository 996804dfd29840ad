"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
library routines on special cases, closed forms, invariants, brute force and
the numbers the pages print.  CPU only."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=16, page_size=4,
                n_pages=12, top_k=5)
    base.update(kw)
    return synth.custom(**base)


def f(bits):
    return synth.bf16_bits_to_f64(bits)


def logical_keys(case):
    """[B][N][P][H][D] float64 keys in logical order (numpy gather)."""
    return f(case.k_pool)[case.page_table]


def logical_values(case):
    return f(case.v_pool)[case.page_table]


# ---------------------------------------------------------------- summaries

def test_summaries_equal_numpy_reduction():
    case = synth.make_case(small())
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table)
    K = logical_keys(case)                       # [B][N][P][H][D]
    np.testing.assert_array_equal(kmin, K.min(axis=2).transpose(0, 2, 1, 3))
    np.testing.assert_array_equal(kmax, K.max(axis=2).transpose(0, 2, 1, 3))


def test_summaries_bound_and_attained():
    case = synth.make_case(small(page_size=8))
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table)
    K = logical_keys(case).transpose(0, 3, 1, 2, 4)   # [B][H][N][P][D]
    assert np.all(K >= kmin[:, :, :, None, :]) and np.all(K <= kmax[:, :, :, None, :])
    assert np.all(np.any(K == kmin[:, :, :, None, :], axis=3))
    assert np.all(np.any(K == kmax[:, :, :, None, :], axis=3))


def test_summaries_reject_bad_page_table():
    case = synth.make_case(small())
    pt = case.page_table.copy()
    pt[0, 3] = case.k_pool.shape[0]
    with pytest.raises(ValueError):
        oracle.summaries(case.k_pool, pt)


# ---------------------------------------------------------------- scores

def _qf(case):
    wl = case.wl
    return f(case.q).reshape(wl.batch, wl.n_kv_heads, wl.group, wl.head_dim)


def test_score_is_upper_bound_of_every_token_dot():
    """mean_h max_t q_h.k_t <= S(p): the score bounds attention logits of the page."""
    case = synth.make_case(small(page_size=8))
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))
    K = logical_keys(case)                                   # [B][N][P][H][D]
    dots = np.einsum("bgjd,bnpgd->bgjnp", _qf(case), K)      # [B][H][G][N][P]
    bound = dots.max(axis=-1).mean(axis=2)                   # [B][H][N]
    assert np.all(s >= bound - 1e-12)


def test_score_is_tight_when_page_tokens_agree():
    """All P tokens equal to the page's first key: S(p) = mean_h q_h.k_0 exactly."""
    case = synth.make_case(small(page_size=8))
    case.k_pool[:] = case.k_pool[:, :1]
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))
    K0 = logical_keys(case)[:, :, 0]                          # [B][N][H][D]
    want = np.einsum("bgjd,bngd->bgjn", _qf(case), K0).mean(axis=2)
    np.testing.assert_allclose(s, want, rtol=0, atol=1e-12)


def test_score_page_size_one_is_group_mean_dot():
    """With one token per page, min = max = k, so S(p) = mean over the group of q_h.k_p."""
    case = synth.make_case(small(page_size=1, n_pages=40))
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))
    K = logical_keys(case)[:, :, 0]                          # [B][N][H][D]
    want = np.einsum("bgjd,bngd->bgjn", _qf(case), K).mean(axis=2)
    np.testing.assert_allclose(s, want, rtol=0, atol=1e-12)


def test_score_symmetric_page_closed_form():
    """A page holding +k and -k has kmax = |k|, kmin = -|k|, so s_h = sum_c |q_hc| |k_c|."""
    wl = small(page_size=2, n_pages=6)
    case = synth.make_case(wl)
    for b in range(wl.batch):
        for p in range(wl.n_pages):
            ph = case.page_table[b, p]
            case.k_pool[ph, 1] = case.k_pool[ph, 0] ^ np.uint16(0x8000)   # exact negation
    s = oracle.scores(case.q, *oracle.summaries(case.k_pool, case.page_table))
    K0 = logical_keys(case)[:, :, 0]                          # [B][N][H][D]
    want = np.einsum("bgjd,bngd->bgjn", np.abs(_qf(case)), np.abs(K0)).mean(axis=2)
    np.testing.assert_allclose(s, want, rtol=0, atol=1e-12)


def test_score_scales_with_query_and_ranking_is_invariant():
    wl = small(n_pages=30, top_k=7)
    case = synth.make_case(wl)
    summ = oracle.summaries(case.k_pool, case.page_table)
    s1 = oracle.scores(case.q, *summ)
    q2 = synth.f64_to_bf16_bits(2.0 * f(case.q))               # exact in bf16
    s2 = oracle.scores(q2, *summ)
    np.testing.assert_array_equal(s2, 2.0 * s1)
    np.testing.assert_array_equal(oracle.topk(s1, wl.top_k), oracle.topk(s2, wl.top_k))


# ---------------------------------------------------------------- top-k

def _brute_topk(s, k):
    """Page p is selected iff fewer than k pages beat it (higher score, or
    equal score and lower id)."""
    n = len(s)
    beats = [sum(1 for j in range(n) if s[j] > s[p] or (s[j] == s[p] and j < p)) for p in range(n)]
    return np.array([p for p in range(n) if beats[p] < k], dtype=np.int32)


def test_topk_equals_rank_counting_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, n + 1))
        s = rng.integers(-4, 5, size=n).astype(np.float64)   # many ties
        np.testing.assert_array_equal(oracle.topk(s, k), _brute_topk(s, k))


def test_topk_is_best_subset_tiny():
    """Exhaustive: the selected set has the largest score sum of all k-subsets,
    and among the sets reaching it the lexicographically smallest ids."""
    rng = np.random.default_rng(6)
    for trial in range(30):
        n = int(rng.integers(2, 9))
        k = int(rng.integers(1, n + 1))
        s = rng.integers(0, 4, size=n).astype(np.float64)
        best = max(itertools.combinations(range(n), k), key=lambda c: (sum(s[list(c)]), [-i for i in c]))
        np.testing.assert_array_equal(oracle.topk(s, k), np.array(best, dtype=np.int32))


def test_topk_contains_argmax_and_prefers_lower_duplicate():
    rng = np.random.default_rng(7)
    s = rng.standard_normal(64)
    sel = oracle.topk(s, 9)
    assert np.argmax(s) in sel
    assert np.all(np.diff(sel) > 0)
    srt = np.sort(s)[::-1]
    s[40] = s[50] = (srt[8] + srt[9]) / 2        # a tie straddling the boundary
    sel = oracle.topk(s, 9)
    assert 40 in sel and 50 not in sel


# ---------------------------------------------------------------- attention

def test_attention_all_pages_equals_sdpa_float64():
    """k = N: sparse attention is dense attention; torch SDPA in float64 agrees."""
    wl = small(n_pages=6, top_k=6, head_dim=32)
    case = synth.make_case(wl)
    sel = np.tile(np.arange(wl.n_pages, dtype=np.int32), (wl.batch, wl.n_kv_heads, 1))
    out = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel)
    K = logical_keys(case).reshape(wl.batch, wl.context, wl.n_kv_heads, wl.head_dim)
    V = logical_values(case).reshape(wl.batch, wl.context, wl.n_kv_heads, wl.head_dim)
    q = torch.from_numpy(f(case.q))[:, :, None, :]                         # [B][Hq][1][D]
    k = torch.from_numpy(K).permute(0, 2, 1, 3).repeat_interleave(wl.group, dim=1)
    v = torch.from_numpy(V).permute(0, 2, 1, 3).repeat_interleave(wl.group, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v)[:, :, 0, :].numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_attention_subset_equals_sdpa_on_gathered_tokens():
    wl = small(n_pages=10, top_k=3, head_dim=16)
    case = synth.make_case(wl)
    rng = np.random.default_rng(3)
    sel = np.sort(np.stack([[rng.choice(wl.n_pages, 3, replace=False) for g in range(wl.n_kv_heads)]
                            for b in range(wl.batch)]), axis=-1).astype(np.int32)
    out = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel, scale=0.3)
    K, V = logical_keys(case), logical_values(case)
    for b in range(wl.batch):
        for h in range(wl.n_q_heads):
            g = h // wl.group
            kk = torch.from_numpy(K[b, sel[b, g], :, g].reshape(-1, wl.head_dim))
            vv = torch.from_numpy(V[b, sel[b, g], :, g].reshape(-1, wl.head_dim))
            qq = torch.from_numpy(f(case.q[b, h]))
            ref = torch.nn.functional.scaled_dot_product_attention(qq[None], kk, vv, scale=0.3)[0]
            np.testing.assert_allclose(out[b, h], ref.numpy(), rtol=0, atol=1e-12)


def test_attention_single_token_returns_its_value():
    wl = small(page_size=1, n_pages=9, top_k=1)
    case = synth.make_case(wl)
    sel = np.full((wl.batch, wl.n_kv_heads, 1), 4, dtype=np.int32)
    out = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel)
    V = logical_values(case)
    for h in range(wl.n_q_heads):
        np.testing.assert_array_equal(out[:, h], V[:, 4, 0, h // wl.group])


def test_attention_identical_keys_or_zero_scale_is_mean_value():
    wl = small(n_pages=8, top_k=3)
    case = synth.make_case(wl)
    sel = np.tile(np.array([1, 4, 6], dtype=np.int32), (wl.batch, wl.n_kv_heads, 1))
    V = logical_values(case)
    mean_v = V[:, [1, 4, 6]].reshape(wl.batch, -1, wl.n_kv_heads, wl.head_dim).mean(axis=1)
    want = np.repeat(mean_v, wl.group, axis=1)
    out0 = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel, scale=0.0)
    np.testing.assert_allclose(out0, want, rtol=0, atol=1e-12)
    case.k_pool[:] = case.k_pool[0, 0]            # every key identical
    out1 = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel)
    np.testing.assert_allclose(out1, want, rtol=0, atol=1e-12)


def test_attention_follows_the_page_table():
    """Permuting physical pages together with the table leaves the result unchanged."""
    wl = small(n_pages=8, top_k=3)
    case = synth.make_case(wl)
    sel = np.tile(np.array([0, 2, 5], dtype=np.int32), (wl.batch, wl.n_kv_heads, 1))
    out = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel)
    perm = np.random.default_rng(1).permutation(case.k_pool.shape[0])
    inv = np.argsort(perm)
    out2 = oracle.attention(case.q, case.k_pool[perm], case.v_pool[perm],
                            inv[case.page_table].astype(np.int32), sel)
    np.testing.assert_array_equal(out, out2)


# ---------------------------------------------------------------- cosine / speculation

def test_group_cosine_closed_forms():
    wl = small()
    case = synth.make_case(wl)
    q = case.q[:1]
    neg = q ^ np.uint16(0x8000)
    np.testing.assert_allclose(oracle.group_cosine(q, q, wl.n_kv_heads), 1.0, atol=1e-12)
    np.testing.assert_allclose(oracle.group_cosine(q, neg, wl.n_kv_heads), -1.0, atol=1e-12)
    a = np.zeros_like(q)
    b = np.zeros_like(q)
    a[..., 0] = synth.f64_to_bf16_bits(1.5)
    b[..., 1] = synth.f64_to_bf16_bits(-2.0)
    np.testing.assert_array_equal(oracle.group_cosine(a, b, wl.n_kv_heads), 0.0)
    np.testing.assert_array_equal(oracle.group_cosine(a, np.zeros_like(q), wl.n_kv_heads), 0.0)
    # group mean: half the heads parallel, half antiparallel -> 0
    mixed = q.copy()
    mixed[0, 1::2] ^= np.uint16(0x8000)
    np.testing.assert_allclose(oracle.group_cosine(q, mixed, wl.n_kv_heads), 0.0, atol=1e-12)


def _trace_case(steps=12, tau=0.8):
    wl = small(n_pages=24, top_k=5, steps=steps, tau=tau, n_jumps=2, head_dim=32)
    case = synth.make_case(wl)
    tr = synth.make_trace(wl, case)
    return wl, case, tr


def test_spec_trace_tau_one_is_plain_selection():
    wl, case, tr = _trace_case()
    res = oracle.speculative_trace(tr.q, case.k_pool, case.v_pool, case.page_table,
                                   wl.n_kv_heads, wl.top_k, tau=1.0)
    assert res["corrected"].all()
    for t in range(wl.steps):
        sel, _, out = oracle.decode_step(tr.q[t], case.k_pool, case.v_pool, case.page_table,
                                         wl.n_kv_heads, wl.top_k)
        np.testing.assert_array_equal(res["sel_used"][t], sel)
        np.testing.assert_array_equal(res["out"][t], out)


def test_spec_trace_never_corrects_below_minus_one():
    wl, case, tr = _trace_case()
    res = oracle.speculative_trace(tr.q, case.k_pool, case.v_pool, case.page_table,
                                   wl.n_kv_heads, wl.top_k, tau=-1.5, with_attention=False)
    assert res["corrected"][0].all() and not res["corrected"][1:].any()
    np.testing.assert_array_equal(res["sel_used"][1:], res["sel_new"][:-1])


def test_spec_trace_jumps_are_corrected_and_reuse_is_previous_selection():
    wl, case, tr = _trace_case(steps=16)
    res = oracle.speculative_trace(tr.q, case.k_pool, case.v_pool, case.page_table,
                                   wl.n_kv_heads, wl.top_k, tau=0.8, with_attention=False)
    for t in tr.jumps:
        assert res["corrected"][t].all()
        assert np.all(res["cbar"][t] < 0.3)
    for t in range(1, wl.steps):
        c = res["corrected"][t]
        np.testing.assert_array_equal(res["sel_used"][t][c], res["sel_new"][t][c])
        np.testing.assert_array_equal(res["sel_used"][t][~c], res["sel_new"][t - 1][~c])
        np.testing.assert_array_equal(c, res["cbar"][t] < 0.8)


# ---------------------------------------------------------------- printed numbers

# ---------------------------------------------------------------- partial pages (decode-time append)

LENS = np.array([37, 9], dtype=np.int32)   # page size 4: 10 and 3 pages started, last ones partial


def test_summaries_with_lengths_equal_numpy_over_written_rows():
    wl = small()
    case = synth.make_case(wl)
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table, seq_len=LENS)
    keys = logical_keys(case)                                    # [B][N][P][H][D]
    P = wl.page_size
    for b, L in enumerate(LENS):
        for p in range(wl.n_pages):
            nt = min(P, max(0, int(L) - p * P))
            if nt == 0:
                assert np.isnan(kmin[b, :, p]).all() and np.isnan(kmax[b, :, p]).all()
                continue
            rows = keys[b, p, :nt]                                # [nt][H][D]
            np.testing.assert_array_equal(kmin[b, :, p], rows.min(axis=0))
            np.testing.assert_array_equal(kmax[b, :, p], rows.max(axis=0))


def test_topk_with_valid_pages_is_brute_force_and_pads():
    rng = np.random.default_rng(4)
    s = np.round(rng.normal(size=(3, 20)), 1)                   # ties likely
    nv = np.array([20, 7, 3])
    sel = oracle.topk(s, 5, nv)
    for u in range(3):
        order = sorted(range(nv[u]), key=lambda p: (-s[u, p], p))
        want = sorted(order[:5]) + [-1] * max(0, 5 - nv[u])
        assert list(sel[u]) == want


def test_attention_with_lengths_equals_sdpa_on_written_tokens():
    wl = small()
    case = synth.make_case(wl)
    P, G = wl.page_size, wl.group
    sel = np.array([[[0, 3, 9], [2, 5, 9]], [[0, 1, 2], [2, 1, 0]]], dtype=np.int32)
    sel = np.sort(sel, axis=-1)
    out = oracle.attention(case.q, case.k_pool, case.v_pool, case.page_table, sel, scale=0.3, seq_len=LENS)
    keys, vals = logical_keys(case), logical_values(case)
    q = torch.from_numpy(f(case.q))
    for b, L in enumerate(LENS):
        for h in range(wl.n_q_heads):
            g = h // G
            rows = [(p, t) for p in sel[b, g] for t in range(min(P, max(0, int(L) - p * P)))]
            kk = torch.from_numpy(np.stack([keys[b, p, t, g] for p, t in rows]))[None]
            vv = torch.from_numpy(np.stack([vals[b, p, t, g] for p, t in rows]))[None]
            ref = torch.nn.functional.scaled_dot_product_attention(q[b, h][None, None], kk, vv, scale=0.3)[0, 0]
            np.testing.assert_allclose(out[b, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_full_lengths_reduce_to_the_length_free_step():
    wl = small()
    case = synth.make_case(wl)
    full = np.full(wl.batch, wl.n_pages * wl.page_size, dtype=np.int32)
    a = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k)
    b_ = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k,
                            seq_len=full)
    for x, y in zip(a, b_):
        np.testing.assert_array_equal(x, y)


def test_append_writes_the_next_row_of_every_head():
    """Appending tokens one at a time from length L0 writes exactly the rows a
    direct copy of the source tokens would, and the summaries over the written
    rows then equal numpy's reduction of those rows."""
    wl = small()
    src = synth.make_case(wl)                                    # the tokens to append
    dst = synth.make_case(small(seed=99))                        # another cache with the same table shape
    P, H, D = wl.page_size, wl.n_kv_heads, wl.head_dim
    lens = np.array([5, 0], dtype=np.int32)
    kp, vp = dst.k_pool, dst.v_pool
    kl, vl = logical_keys(src), logical_values(src)
    want_k, want_v = f(kp).copy(), f(vp).copy()
    for step in range(11):
        k_new = np.stack([src.k_pool[src.page_table[b, (lens[b] // P)], lens[b] % P] for b in range(wl.batch)])
        v_new = np.stack([src.v_pool[src.page_table[b, (lens[b] // P)], lens[b] % P] for b in range(wl.batch)])
        for b in range(wl.batch):
            t = int(lens[b])
            want_k[dst.page_table[b, t // P], t % P] = kl[b, t // P, t % P]
            want_v[dst.page_table[b, t // P], t % P] = vl[b, t // P, t % P]
        kp, vp, lens2 = oracle.append(kp, vp, dst.page_table, lens, k_new, v_new)
        np.testing.assert_array_equal(lens2, lens + 1)
        lens = lens2
        np.testing.assert_array_equal(f(kp), want_k)
        np.testing.assert_array_equal(f(vp), want_v)
    kmin, kmax = oracle.summaries(kp, dst.page_table, seq_len=lens)
    for b, L in enumerate(lens):
        rows = f(kp)[dst.page_table[b]].reshape(-1, H, D)[:L]   # logical token order
        last = (L - 1) // P
        np.testing.assert_array_equal(kmin[b, :, last], rows[last * P:L].min(axis=0))
        np.testing.assert_array_equal(kmax[b, :, last], rows[last * P:L].max(axis=0))


# ---------------------------------------------------------------- several queries per step

def _brute_topk_valid(s, k, started):
    """Top-k over each sequence's started pages by a full sort (ties to the
    lower id), ascending, -1 padded: [B][H][k]."""
    B, H, N = s.shape
    out = np.full((B, H, k), -1, dtype=np.int32)
    for b in range(B):
        for g in range(H):
            n = int(started[b])
            order = sorted(range(n), key=lambda p: (-s[b, g, p], p))[:k]
            out[b, g, :len(order)] = sorted(order)
    return out


def _multi_case(T=3, **kw):
    wl = small(**kw)
    case = synth.make_case(wl)
    rng = np.random.default_rng(123)
    qs = synth.f64_to_bf16_bits(rng.standard_normal((wl.batch, T, wl.n_q_heads, wl.head_dim)))
    lens = np.array([wl.n_pages * wl.page_size - 3, 2 * wl.page_size + 1], dtype=np.int32)[:wl.batch]
    return wl, case, qs, lens


def test_multi_query_with_one_query_is_the_decode_step():
    wl, case, qs, lens = _multi_case(T=1)
    sel, s, out = oracle.multi_query_step(qs, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads,
                                          wl.top_k, lens)
    ref = oracle.decode_step(qs[:, 0], case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k,
                             seq_len=lens)
    np.testing.assert_array_equal(sel, ref[0])
    np.testing.assert_array_equal(s, ref[1])
    np.testing.assert_array_equal(out[:, 0], ref[2])


def test_multi_query_score_is_the_mean_over_the_wider_group():
    """The step's score equals the single-query score of a KV head whose
    group holds all T x G query rows (one call, one mean)."""
    wl, case, qs, lens = _multi_case(T=3)
    B, T, Hq, D = qs.shape
    H, G = wl.n_kv_heads, wl.group
    sel, s, _ = oracle.multi_query_step(qs, case.k_pool, case.v_pool, case.page_table, H, wl.top_k, lens)
    wide = qs.reshape(B, T, H, G, D).transpose(0, 2, 1, 3, 4).reshape(B, H * T * G, D)
    summ = oracle.summaries(case.k_pool, case.page_table, seq_len=lens)
    s_wide = oracle.scores(wide, *summ)
    np.testing.assert_allclose(s, s_wide, rtol=1e-12, atol=1e-12)
    started = (lens + wl.page_size - 1) // wl.page_size
    np.testing.assert_array_equal(sel, _brute_topk_valid(s_wide, wl.top_k, started))


def test_multi_query_attention_is_causal_sdpa():
    """Query tau of sequence b attends over the selected tokens at positions
    below L - T + tau + 1 (float64 SDPA on the gathered tokens)."""
    wl, case, qs, lens = _multi_case(T=3)
    B, T, Hq, D = qs.shape
    P, G = wl.page_size, wl.group
    sel, _, out = oracle.multi_query_step(qs, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads,
                                          wl.top_k, lens, scale=0.25)
    keys, vals = logical_keys(case), logical_values(case)
    for b, L in enumerate(lens):
        for t in range(T):
            limit = int(L) - T + t + 1
            for h in range(Hq):
                g = h // G
                rows = [(p, r) for p in sel[b, g] if p >= 0 for r in range(P) if p * P + r < limit]
                assert rows, "a query with no token to attend"
                kk = torch.from_numpy(np.stack([keys[b, p, r, g] for p, r in rows]))[None]
                vv = torch.from_numpy(np.stack([vals[b, p, r, g] for p, r in rows]))[None]
                qq = torch.from_numpy(f(qs[b, t, h]))[None, None]
                ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=0.25)[0, 0]
                np.testing.assert_allclose(out[b, t, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_multi_query_later_tokens_stay_out_of_earlier_queries():
    """Changing the value of each sequence's newest token changes only the
    last query's output (every page selected, so that token is read)."""
    wl, case, qs, lens = _multi_case(T=3, top_k=12)
    T = qs.shape[1]
    args = (case.k_pool, case.page_table, wl.n_kv_heads, wl.top_k, lens)
    _, _, out = oracle.multi_query_step(qs, case.k_pool, case.v_pool, *args[1:])
    v2 = np.array(case.v_pool, copy=True)
    P = wl.page_size
    for b, L in enumerate(lens):
        v2[case.page_table[b, (L - 1) // P], (L - 1) % P] ^= 0x0040     # flip a mantissa bit of every channel
    _, _, out2 = oracle.multi_query_step(qs, case.k_pool, v2, *args[1:])
    np.testing.assert_array_equal(out[:, :T - 1], out2[:, :T - 1])
    assert np.all(np.abs(out[:, T - 1] - out2[:, T - 1]).max(axis=-1) > 0)


def test_kv_cache_size_matches_printed_llama65b_figure():
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_size_llama65b.json")))
    n = oracle.kv_cache_bytes(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["n_tokens"], g["bytes_per_elem"])
    assert abs(n / 1e9 - g["stated_gb"]) <= g["stated_rounding_gb"]
