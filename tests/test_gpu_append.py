"""Decode-time append and partial last pages through the C ABI, against the
oracle: appended rows and incrementally kept summaries bit-exact, selection
over started pages bit-exact, attention over written tokens within the
tolerance, for page sizes 16, 32 and 64."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    kvr.kvr_get_status()
    yield
    assert kvr.kvr_get_status() == 0


# (page size, lengths, top-k): last pages partial; with P = 64 the second
# chunk of a partial page is empty (276 tokens) or partial (114)
CASES = [(16, [300, 37], 6), (32, [300, 70], 5), (64, [276, 114], 3)]


def workload(P, k):
    return synth.custom(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=P,
                        n_pages=640 // P, top_k=k)


def dev_summaries(dc, seq_len):
    wl = dc.wl
    summ = torch.zeros((wl.batch, wl.n_kv_heads, wl.n_pages, 2, wl.head_dim), dtype=torch.int16, device="cuda")
    kvr.kvr_build_summaries_len(dc.dims, dc.k_pool, dc.page_table, seq_len, summ)
    return summ


def check_summaries(summ_dev, kmin, kmax, lens, P):
    s = gh.f64(summ_dev)
    for b, L in enumerate(lens):
        n = (int(L) + P - 1) // P
        np.testing.assert_array_equal(s[b, :, :n, 0], kmin[b, :, :n])
        np.testing.assert_array_equal(s[b, :, :n, 1], kmax[b, :, :n])


@pytest.mark.parametrize("P,lens,k", CASES)
def test_summaries_over_written_tokens(P, lens, k):
    wl = workload(P, k)
    case = synth.make_case(wl)
    dc = gh.DevCase(case)
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table, seq_len=np.array(lens))
    check_summaries(dev_summaries(dc, L), kmin, kmax, lens, P)


@pytest.mark.parametrize("P,lens,k", CASES)
def test_append_matches_oracle(P, lens, k):
    """40 appends per sequence: pools and lengths bit-exact, the summaries kept
    by the appends equal the oracle's summaries over the written tokens."""
    wl = workload(P, k)
    case = synth.make_case(wl)
    new = synth.make_case(synth.custom(**{**wl.__dict__, "name": "new", "seed": 123}))
    dc = gh.DevCase(case)
    lens = np.array(lens, dtype=np.int32)
    L = torch.tensor(lens, device="cuda")
    summ = dev_summaries(dc, L)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    for step in range(40):
        # the new rows: a token of the other cache per (sequence, head)
        k_new = np.stack([new.k_pool[new.page_table[b, step // P], step % P] for b in range(wl.batch)])
        v_new = np.stack([new.v_pool[new.page_table[b, step // P], step % P] for b in range(wl.batch)])
        kvr.kvr_append_kv(dc.dims, gh.t16(k_new), gh.t16(v_new), dc.page_table, L, dc.k_pool, dc.v_pool, summ)
        kp, vp, lens = oracle.append(kp, vp, case.page_table, lens, k_new, v_new)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(L.cpu().numpy(), lens)
    np.testing.assert_array_equal(gh.bits(dc.k_pool), kp)
    np.testing.assert_array_equal(gh.bits(dc.v_pool), vp)
    kmin, kmax = oracle.summaries(kp, case.page_table, seq_len=lens)
    check_summaries(summ, kmin, kmax, lens, P)


def test_append_to_a_full_sequence_is_refused_and_reported():
    wl = workload(16, 4)
    case = synth.make_case(wl)
    dc = gh.DevCase(case)
    full = wl.n_pages * wl.page_size
    L = torch.tensor([full, 5], dtype=torch.int32, device="cuda")
    summ = dev_summaries(dc, L)
    before = gh.bits(dc.k_pool).copy()
    rows = gh.t16(np.zeros((wl.batch, wl.n_kv_heads, wl.head_dim), dtype=np.uint16))
    kvr.kvr_append_kv(dc.dims, rows, rows, dc.page_table, L, dc.k_pool, dc.v_pool, summ)
    assert kvr.kvr_get_status() & kvr.KVR_ST_BAD_INDEX
    np.testing.assert_array_equal(L.cpu().numpy(), [full, 6])
    after = gh.bits(dc.k_pool)
    phys = case.page_table[1, 0]
    changed = np.argwhere(after != before)
    assert len(changed) and np.all(changed[:, 0] == phys) and np.all(changed[:, 1] == 5)


@pytest.mark.parametrize("P,lens,k", CASES)
def test_selection_and_attention_over_written_tokens(P, lens, k):
    wl = workload(P, k)
    case = synth.make_case(wl)
    dc = gh.DevCase(case)
    lens_np = np.array(lens, dtype=np.int32)
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    summ = dev_summaries(dc, L)
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table,
                                             wl.n_kv_heads, k, seq_len=lens_np)
    sel = torch.full((wl.batch, wl.n_kv_heads, k), -7, dtype=torch.int32, device="cuda")
    sel_phys = torch.full_like(sel, -7)
    ws = gh.workspace(dc.dims, k, kvr.KVR_OP_SELECT)
    kvr.kvr_select_pages_len(dc.dims, dc.q, summ, dc.page_table, L, k, sel, sel_phys, None, ws, ws.numel())
    np.testing.assert_array_equal(sel.cpu().numpy(), sel_ref)
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    wa = gh.workspace(dc.dims, k, kvr.KVR_OP_ATTN)
    kvr.kvr_sparse_decode_attn_len(dc.dims, dc.q, dc.k_pool, dc.v_pool, dc.page_table, L, sel_phys, k, 0.0, out,
                                   wa, wa.numel())
    gh.assert_attn_close(out.cpu().numpy(), out_ref)


def test_fewer_started_pages_than_k_pads_and_attends_over_them():
    """A 20-token sequence of 16-token pages has 2 pages: with k = 5 its rows are
    [0, 1, -1, -1, -1] and attention runs over its 20 tokens."""
    wl = workload(16, 5)
    case = synth.make_case(wl)
    dc = gh.DevCase(case)
    lens_np = np.array([20, 300], dtype=np.int32)
    L = torch.tensor(lens_np, device="cuda")
    summ = dev_summaries(dc, L)
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table,
                                             wl.n_kv_heads, 5, seq_len=lens_np)
    assert (sel_ref[0] == np.array([0, 1, -1, -1, -1])).all()
    sel = torch.full((wl.batch, wl.n_kv_heads, 5), -7, dtype=torch.int32, device="cuda")
    sel_phys = torch.full_like(sel, -7)
    ws = gh.workspace(dc.dims, 5, kvr.KVR_OP_SELECT)
    kvr.kvr_select_pages_len(dc.dims, dc.q, summ, dc.page_table, L, 5, sel, sel_phys, None, ws, ws.numel())
    np.testing.assert_array_equal(sel.cpu().numpy()[0], sel_ref[0])
    assert (sel_phys.cpu().numpy()[0, :, 2:] == -1).all()
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    wa = gh.workspace(dc.dims, 5, kvr.KVR_OP_ATTN)
    phys_ref = np.where(sel_ref >= 0, np.take_along_axis(case.page_table[:, None, :].repeat(2, 1),
                                                         np.maximum(sel_ref, 0), axis=2), -1).astype(np.int32)
    kvr.kvr_sparse_decode_attn_len(dc.dims, dc.q, dc.k_pool, dc.v_pool, dc.page_table, L,
                                   torch.from_numpy(phys_ref).cuda(), 5, 0.0, out, wa, wa.numel())
    gh.assert_attn_close(out.cpu().numpy()[0], out_ref[0])


def test_decode_loop_append_select_attend():
    """Eight decode steps of a growing cache: append the step's token, select
    over the started pages, attend over the written tokens; the selection is
    compared where the oracle's top-k margin is clear, the attention of the
    GPU's own selection always."""
    P, k = 16, 4
    wl = workload(P, k)
    case = synth.make_case(wl)
    new = synth.make_case(synth.custom(**{**wl.__dict__, "name": "new", "seed": 321}))
    dc = gh.DevCase(case)
    lens = np.array([45, 17], dtype=np.int32)
    L = torch.tensor(lens, device="cuda")
    summ = dev_summaries(dc, L)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    ws = gh.workspace(dc.dims, k, kvr.KVR_OP_SELECT)
    wa = gh.workspace(dc.dims, k, kvr.KVR_OP_ATTN)
    compared = 0
    for step in range(8):
        k_new = np.stack([new.k_pool[new.page_table[b, step], 0] for b in range(wl.batch)])
        v_new = np.stack([new.v_pool[new.page_table[b, step], 0] for b in range(wl.batch)])
        q = new.q if step % 2 else case.q
        kvr.kvr_append_kv(dc.dims, gh.t16(k_new), gh.t16(v_new), dc.page_table, L, dc.k_pool, dc.v_pool, summ)
        kp, vp, lens = oracle.append(kp, vp, case.page_table, lens, k_new, v_new)
        sel = torch.empty((wl.batch, wl.n_kv_heads, k), dtype=torch.int32, device="cuda")
        sel_phys = torch.empty_like(sel)
        kvr.kvr_select_pages_len(dc.dims, gh.t16(q), summ, dc.page_table, L, k, sel, sel_phys, None, ws, ws.numel())
        out = torch.empty((wl.batch, wl.n_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
        kvr.kvr_sparse_decode_attn_len(dc.dims, gh.t16(q), dc.k_pool, dc.v_pool, dc.page_table, L, sel_phys, k,
                                       0.0, out, wa, wa.numel())
        sel_gpu = sel.cpu().numpy()
        sel_ref, s, _ = oracle.decode_step(q, kp, vp, case.page_table, wl.n_kv_heads, k, seq_len=lens)
        nv = oracle.valid_pages(lens, P)
        for b in range(wl.batch):
            for g in range(wl.n_kv_heads):
                row = np.sort(s[b, g, :nv[b]])[::-1]
                if len(row) <= k or row[k - 1] - row[k] >= 1e-4:
                    np.testing.assert_array_equal(sel_gpu[b, g], sel_ref[b, g])
                    compared += 1
        ref = oracle.attention(q, kp, vp, case.page_table, sel_gpu, seq_len=lens)
        gh.assert_attn_close(out.cpu().numpy(), ref)
    assert compared >= 24


@pytest.mark.parametrize("n_q_heads,n_kv_heads", [(8, 8), (16, 2)], ids=["G1", "G8"])
def test_lengths_for_other_group_sizes(n_q_heads, n_kv_heads):
    """G = 1 (spare residual columns mostly empty) and G = 8 (the residual in
    a second MMA) with a partial last page and a sequence shorter than k."""
    wl = synth.custom(batch=2, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=128, page_size=32,
                      n_pages=20, top_k=5)
    case = synth.make_case(wl)
    dc = gh.DevCase(case)
    lens_np = np.array([300, 70], dtype=np.int32)
    L = torch.tensor(lens_np, device="cuda")
    summ = dev_summaries(dc, L)
    sel_ref, _, out_ref = oracle.decode_step(case.q, case.k_pool, case.v_pool, case.page_table,
                                             wl.n_kv_heads, 5, seq_len=lens_np)
    sel = torch.full((wl.batch, wl.n_kv_heads, 5), -7, dtype=torch.int32, device="cuda")
    sel_phys = torch.full_like(sel, -7)
    ws = gh.workspace(dc.dims, 5, kvr.KVR_OP_SELECT)
    kvr.kvr_select_pages_len(dc.dims, dc.q, summ, dc.page_table, L, 5, sel, sel_phys, None, ws, ws.numel())
    np.testing.assert_array_equal(sel.cpu().numpy(), sel_ref)
    out = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    wa = gh.workspace(dc.dims, 5, kvr.KVR_OP_ATTN)
    kvr.kvr_sparse_decode_attn_len(dc.dims, dc.q, dc.k_pool, dc.v_pool, dc.page_table, L, sel_phys, 5, 0.0, out,
                                   wa, wa.numel())
    gh.assert_attn_close(out.cpu().numpy(), out_ref)


def accept_started(lens, P, k):
    """Row b's query is kept when its top-k boundary among the sequence's
    started pages (summaries over the written tokens) has a margin of at
    least the oracle's, so that the fp32 and fp64 selections agree."""
    def accept(case, b):
        nv = -(-int(lens[b]) // P)
        if nv <= k:  # every started page is selected: no boundary
            return True
        summ = oracle.summaries(case.k_pool, case.page_table[b:b + 1], seq_len=lens[b:b + 1])
        s = oracle.scores(case.q[b:b + 1], *summ)[..., :nv]
        return bool(np.all(oracle.topk_margin(s, k) >= oracle.MARGIN))
    return accept


@pytest.mark.parametrize("n_pages", [1500, 3000, 5000, 9000])
def test_lengths_at_the_larger_top_k_shapes(n_pages):
    """Selection over started pages at the page counts of the top-k's larger
    shapes (256 threads x 8 keys, 512 x 8, 512 x 16, 1024 x 16): a full
    sequence, one ending inside a page halfway, and one with fewer started
    pages than k (its last slots -1)."""
    P, k = 16, 64
    lens = np.array([n_pages * P, n_pages * P // 2 + 5, 40 * P - 3], dtype=np.int32)
    wl = synth.custom(batch=3, n_q_heads=4, n_kv_heads=1, head_dim=128, page_size=P, n_pages=n_pages, top_k=k)
    case = synth.make_case(wl, accept=accept_started(lens, P, k))
    dc = gh.DevCase(case)
    L = torch.tensor(lens, device="cuda")
    summ = dev_summaries(dc, L)
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table, seq_len=lens)
    check_summaries(summ, kmin, kmax, lens, P)
    sel_ref = oracle.topk(oracle.scores(case.q, kmin, kmax), k, n_valid=oracle.valid_pages(lens, P)[:, None])
    assert (sel_ref[2, 0, 40:] == -1).all() and (sel_ref[2, 0, :40] == np.arange(40)).all()
    sel = torch.full((wl.batch, wl.n_kv_heads, k), -7, dtype=torch.int32, device="cuda")
    sel_phys = torch.full_like(sel, -7)
    ws = gh.workspace(dc.dims, k, kvr.KVR_OP_SELECT)
    kvr.kvr_select_pages_len(dc.dims, dc.q, summ, dc.page_table, L, k, sel, sel_phys, None, ws, ws.numel())
    np.testing.assert_array_equal(sel.cpu().numpy(), sel_ref)
    phys_ref = np.where(sel_ref >= 0, np.take_along_axis(case.page_table[:, None, :], np.maximum(sel_ref, 0),
                                                         axis=2), -1)
    np.testing.assert_array_equal(sel_phys.cpu().numpy(), phys_ref)
