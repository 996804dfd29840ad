"""Several query tokens per sequence in one step, through the C ABI, against
the oracle (oracle.multi_query_step): the step's selection bit-exact (the
generator keeps a top-k margin of the mean page score over the step's query
rows), the causal attention of every query token within the tolerance, in
fp32 and in bf16; at the Llama-3.1-8B layer shapes for T = 2 and 4, and on
small shapes for every supported number of query rows (G T = 1 .. 16) and
page size, with partial last pages."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_page_build_b300 import kvr, synth
from tests import gpuhelp as gh

pytestmark = pytest.mark.gpu

BF16_REL = 2.0 ** -8      # the output's rounding to bf16 adds at most 2^-9 |o|


@pytest.fixture(autouse=True)
def _status_clean():
    kvr.kvr_get_status()
    yield
    assert kvr.kvr_get_status() == 0


def make(wl, T, lens, rho=0.9):
    """The case, its T queries per sequence (redrawn until the step's score
    keeps the margin) and the oracle's step."""
    case = synth.make_case(wl)
    lens = np.asarray(lens, dtype=np.int32)
    summ = oracle.summaries(case.k_pool, case.page_table, seq_len=lens)
    qs = synth.make_multi_queries(case, T, oracle.accept_multi_query(summ, wl.n_kv_heads, wl.top_k, lens,
                                                                    wl.page_size), rho=rho)
    ref = oracle.multi_query_step(qs, case.k_pool, case.v_pool, case.page_table, wl.n_kv_heads, wl.top_k, lens,
                                  summ=summ)
    return case, qs, lens, ref


def run(case, qs, lens, T, out_dtype=kvr.KVR_DTYPE_F32, dc=None):
    wl = case.wl
    dc = dc or gh.DevCase(case)
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    summ = torch.zeros((wl.batch, wl.n_kv_heads, wl.n_pages, 2, wl.head_dim), dtype=torch.int16, device="cuda")
    kvr.kvr_build_summaries_len(dc.dims, dc.k_pool, dc.page_table, L, summ)
    k = wl.top_k
    sel = torch.full((wl.batch, wl.n_kv_heads, k), -7, dtype=torch.int32, device="cuda")
    sel_phys = torch.full_like(sel, -7)
    scores = torch.full((wl.batch, wl.n_kv_heads, wl.n_pages), float("nan"), dtype=torch.float32, device="cuda")
    q = gh.t16(qs)
    ws = gh.workspace(dc.dims, k, kvr.KVR_OP_SELECT)
    kvr.kvr_select_pages_multi(dc.dims, q, T, summ, dc.page_table, L, k, sel, sel_phys, scores, ws, ws.numel())
    shape = (wl.batch, T, wl.n_q_heads, wl.head_dim)
    out = (torch.full(shape, float("nan"), dtype=torch.float32, device="cuda") if out_dtype == kvr.KVR_DTYPE_F32
           else torch.full(shape, -1, dtype=torch.int16, device="cuda"))
    wa = gh.workspace(dc.dims, k, kvr.KVR_OP_ATTN)
    kvr.kvr_sparse_decode_attn_multi(dc.dims, q, T, dc.k_pool, dc.v_pool, dc.page_table, L, sel, sel_phys, k, 0.0,
                                     out, out_dtype, wa, wa.numel())
    torch.cuda.synchronize()
    return sel.cpu().numpy(), sel_phys.cpu().numpy(), scores.cpu().numpy(), out


def score_bound(qs, kmin, kmax, n_kv_heads):
    """|fp32 score - exact| for a mean over R = T G query rows: at most
    (8 + log2 R + 4) rounded additions over terms whose magnitudes sum to
    A = sum over rows and channels of |q| max(|kmin|, |kmax|), divided by R."""
    B, T, Hq, D = qs.shape
    G = Hq // n_kv_heads
    R = T * G
    qa = np.abs(synth.bf16_bits_to_f64(qs)).reshape(B, T, n_kv_heads, G, D).transpose(0, 2, 1, 3, 4)
    ka = np.nan_to_num(np.maximum(np.abs(kmin), np.abs(kmax)))
    A = np.einsum("bhtjd,bhnd->bhn", qa, ka)
    return (8 + int(np.log2(R)) + 4) * 2.0 ** -24 * A / R + 1e-30


def check(case, qs, lens, ref, sel, sel_phys, scores, out, out_dtype=kvr.KVR_DTYPE_F32):
    wl = case.wl
    sel_ref, s_ref, out_ref = ref
    np.testing.assert_array_equal(sel, sel_ref)
    phys_ref = np.where(sel_ref >= 0, np.take_along_axis(case.page_table[:, None, :],
                                                          np.maximum(sel_ref, 0), axis=2), -1)
    np.testing.assert_array_equal(sel_phys, phys_ref)
    kmin, kmax = oracle.summaries(case.k_pool, case.page_table, seq_len=lens)
    started = oracle.valid_pages(lens, wl.page_size)
    for b in range(wl.batch):
        n = int(started[b])
        err = np.abs(scores[b, :, :n] - s_ref[b, :, :n])
        assert np.all(err <= score_bound(qs[b:b + 1], kmin[b:b + 1, :, :n], kmax[b:b + 1, :, :n],
                                         wl.n_kv_heads)[0]), float(err.max())
    if out_dtype == kvr.KVR_DTYPE_F32:
        gh.assert_attn_close(out.cpu().numpy(), out_ref)
    else:
        o = gh.f64(out)
        assert np.all(np.abs(o - out_ref) <= gh.ATOL + BF16_REL * np.abs(out_ref)), float(np.abs(o - out_ref).max())


@pytest.mark.parametrize("T", [2, 4])
def test_llama_shapes_several_queries(T):
    """The Llama-3.1-8B layer (8 sequences, 32/8 heads, 1024 pages of 32,
    top-k 64) with T = 2 and 4 query tokens (8 and 16 query rows per KV
    head); the sequences end inside their last page."""
    wl = synth.WORKLOADS[2]
    lens = wl.n_pages * wl.page_size - np.array([0, 1, 5, 17, 31, 32, 33, 300])
    case, qs, lens, ref = make(wl, T, lens)
    check(case, qs, lens, ref, *run(case, qs, lens, T))


def test_repeated_several_query_steps_on_one_workspace():
    """The selection and the causal attention of a step of 4 queries, run
    eight times back to back on one workspace, each time against the oracle:
    the attention is resident while the selection still writes the logical
    ids it reads (programmatic dependent launch), so it reads them at L2."""
    wl = synth.WORKLOADS[2]
    lens = wl.n_pages * wl.page_size - np.array([0, 1, 5, 17, 31, 32, 33, 300])
    T = 4
    case, qs, lens, ref = make(wl, T, lens)
    dc = gh.DevCase(case)
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    summ = torch.zeros((wl.batch, wl.n_kv_heads, wl.n_pages, 2, wl.head_dim), dtype=torch.int16, device="cuda")
    kvr.kvr_build_summaries_len(dc.dims, dc.k_pool, dc.page_table, L, summ)
    k = wl.top_k
    q = gh.t16(qs)
    ws = gh.workspace(dc.dims, k, kvr.KVR_OP_STEP)
    first = None
    for rep in range(8):
        sel = torch.full((wl.batch, wl.n_kv_heads, k), -7, dtype=torch.int32, device="cuda")
        sel_phys = torch.full_like(sel, -7)
        out = torch.full((wl.batch, T, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
        kvr.kvr_select_pages_multi(dc.dims, q, T, summ, dc.page_table, L, k, sel, sel_phys, None, ws, ws.numel())
        kvr.kvr_sparse_decode_attn_multi(dc.dims, q, T, dc.k_pool, dc.v_pool, dc.page_table, L, sel, sel_phys, k, 0.0,
                                         out, kvr.KVR_DTYPE_F32, ws, ws.numel())
        torch.cuda.synchronize()
        np.testing.assert_array_equal(sel.cpu().numpy(), ref[0], err_msg=f"run {rep}")
        if first is None:
            gh.assert_attn_close(out.cpu().numpy(), ref[2])
            first = out.clone()
        else:
            assert torch.equal(out, first), f"run {rep}"


@pytest.mark.parametrize("T", [1, 2, 4])
def test_bf16_output_is_the_fp32_output_rounded(T):
    """KVR_DTYPE_BF16 stores the fp32 result rounded to nearest even once:
    bit-equal to rounding the fp32 output on the host, and within
    2e-3 + 2^-8 |o| of the oracle."""
    wl = synth.custom(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=32, n_pages=64, top_k=12)
    lens = [64 * 32 - 7, 40 * 32 + 3]
    case, qs, lens, ref = make(wl, T, lens)
    dc = gh.DevCase(case)
    res32 = run(case, qs, lens, T, kvr.KVR_DTYPE_F32, dc=dc)
    res16 = run(case, qs, lens, T, kvr.KVR_DTYPE_BF16, dc=dc)
    check(case, qs, lens, ref, *res16, out_dtype=kvr.KVR_DTYPE_BF16)
    o32 = res32[3].cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(gh.bits(res16[3]), synth.f64_to_bf16_bits(o32))


# (G, T, page size): every supported number of query rows G T; T > P makes
# whole chunks invisible to the earlier query tokens
SWEEP = [(1, 2, 16), (2, 2, 32), (4, 2, 64), (8, 2, 16), (4, 4, 32), (2, 8, 64), (1, 16, 16), (8, 1, 32),
         (1, 8, 32), (2, 4, 16)]


@pytest.mark.parametrize("G,T,P", SWEEP)
def test_rows_and_page_sizes(G, T, P):
    H = 2
    wl = synth.custom(batch=2, n_q_heads=G * H, n_kv_heads=H, head_dim=128, page_size=P, n_pages=1024 // P,
                      top_k=max(3, 160 // P))
    lens = [1024 - 3, 9 * P + T - 1]
    case, qs, lens, ref = make(wl, T, lens)
    check(case, qs, lens, ref, *run(case, qs, lens, T))


def test_one_query_equals_the_length_path():
    """T = 1 is kvr_sparse_decode_attn_len with a choice of output type: the
    fp32 outputs are bit-identical."""
    wl = synth.custom(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=32, n_pages=64, top_k=12)
    lens = [64 * 32 - 9, 23 * 32 + 1]
    case, qs, lens, ref = make(wl, 1, lens)
    dc = gh.DevCase(case)
    sel, sel_phys, _, out = run(case, qs, lens, 1, dc=dc)
    L = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out_len = torch.full((wl.batch, wl.n_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    wa = gh.workspace(dc.dims, wl.top_k, kvr.KVR_OP_ATTN)
    kvr.kvr_sparse_decode_attn_len(dc.dims, gh.t16(qs[:, 0]), dc.k_pool, dc.v_pool, dc.page_table, L,
                                   torch.from_numpy(sel_phys).cuda(), wl.top_k, 0.0, out_len, wa, wa.numel())
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], out_len)


def test_newest_token_reaches_only_the_last_query():
    """Changing the K and V of each sequence's newest token changes the
    output of the step's last query token only; the earlier ones are
    bit-identical (they may not see it)."""
    T = 4
    wl = synth.custom(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, page_size=32, n_pages=64, top_k=64)
    lens = [64 * 32 - 5, 40 * 32 + 2]
    case, qs, lens, ref = make(wl, T, lens)
    dc = gh.DevCase(case)
    _, _, _, out_a = run(case, qs, lens, T, dc=dc)
    sign = torch.tensor(-32768, dtype=torch.int16, device="cuda")   # the bf16 sign bit
    for b, L in enumerate(lens):                    # top_k = N: every started page is selected
        phys, row = int(case.page_table[b, (L - 1) // 32]), int((L - 1) % 32)
        dc.k_pool[phys, row] ^= sign                # K and V of the newest token negated (finite)
        dc.v_pool[phys, row] ^= sign
    _, _, _, out_b = run(case, qs, lens, T, dc=dc)
    assert torch.equal(out_a[:, :T - 1], out_b[:, :T - 1])
    assert not torch.equal(out_a[:, T - 1], out_b[:, T - 1])
